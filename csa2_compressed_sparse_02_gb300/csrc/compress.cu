// Compressor + NVFP4 cache append + FP8 ring window write.
// "DeepSeek-V4.1-Flash-NVFP4" §3.2 (2:1 softmax-gated pooling, NVFP4 with one
// E4M3 scale per 16 elements, pending half-pair kept during decode) and §3.1
// (128-slot FP8 ring, one write per token).
//
// Work split: one CTA of 128 threads owns one sequence's slice of pairs; each
// thread owns 4 consecutive channels, so one NVFP4 group of 16 channels is 4
// adjacent lanes and its amax is two xor-shuffles away. Memory-bound and tiny
// at decode (one token per sequence); at prefill the pairs are spread over
// CTAs of 16 pairs each.
#include "common.cuh"
#include "sm100.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 128;   // 128 x 4 channels = D
constexpr int kPairsPerCta = 16;

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// Softmax over the pair of gate logits, per channel; fp32 with the IEEE divide.
__device__ __forceinline__ float pool1(float k0, float k1, float g0, float g1) {
    float m = fmaxf(g0, g1);
    float e0 = expf(g0 - m), e1 = expf(g1 - m);
    return __fdiv_rn(__fmaf_rn(e0, k0, __fmul_rn(e1, k1)), __fadd_rn(e0, e1));
}

// NVFP4 for the 4 channels this thread holds; the 16-channel group spans lanes
// 4k..4k+3. Returns 4 codes packed as 2 bytes (element 0 in the low nibble)
// and the group's E4M3 scale byte. Every lane of the warp must call this.
__device__ __forceinline__ uint32_t nvfp4_4(float4 c, uint8_t& scale_byte) {
    float amax = fmaxf(fmaxf(fabsf(c.x), fabsf(c.y)), fmaxf(fabsf(c.z), fabsf(c.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    uint8_t sb = e4m3_byte(__fdiv_rn(amax, 6.0f));
    float S = e4m3_value(sb);
    scale_byte = sb;
    if (S == 0.0f) return 0u;
    return e2m1_code_rne(__fdiv_rn(c.x, S)) | (e2m1_code_rne(__fdiv_rn(c.y, S)) << 4) |
           (e2m1_code_rne(__fdiv_rn(c.z, S)) << 8) | (e2m1_code_rne(__fdiv_rn(c.w, S)) << 12);
}

// Rotary embedding of a compressed row ("CSA2稀疏注意力、384专家MoE与1M上下文" §2.2
// compress_rope_theta, §四 rope_scaling yarn; "DeepSeek-V4.1-Flash-NVFP4" §3.2).
// The last `dim` channels turn in adjacent pairs by pos * theta_i, theta_i the
// YaRN frequency (Peng et al. 2023, NTK-by-parts) of the RoFormer frequency
// base^(-2i/dim). fp64 throughout; the caller rounds the result to fp32.
struct RopeArgs {
    int dim;  // 0: no rotation
    double base, factor, orig_len, beta_fast, beta_slow;
};

__device__ __forceinline__ double yarn_freq(int i, const RopeArgs& r) {
    const double f = pow(r.base, -(double)(2 * i) / (double)r.dim);
    // turns of this pair over the original context: orig_len / (2 pi / f)
    const double turns = r.orig_len * f * 0.15915494309189535;  // 1 / (2 pi)
    double keep;  // share of the unscaled frequency
    if (turns > r.beta_fast) keep = 1.0;
    else if (turns < r.beta_slow) keep = 0.0;
    else keep = (turns - r.beta_slow) / (r.beta_fast - r.beta_slow);
    return f * keep + (f / r.factor) * (1.0 - keep);
}

// Rotates channels ch..ch+3 of a row at raw position pos when they fall in the
// rotated tail (ch and dim multiples of 4, so a pair never straddles threads).
__device__ __forceinline__ float4 rope4(float4 v, int ch, int64_t pos, const RopeArgs& r) {
    const int first = kD - r.dim;
    if (r.dim <= 0 || ch < first) return v;
    const int i0 = (ch - first) >> 1;
    double s0, c0, s1, c1;
    sincos((double)pos * yarn_freq(i0, r), &s0, &c0);
    sincos((double)pos * yarn_freq(i0 + 1, r), &s1, &c1);
    const double x = v.x, y = v.y, z = v.z, w = v.w;
    return make_float4((float)(x * c0 - y * s0), (float)(x * s0 + y * c0),
                       (float)(z * c1 - w * s1), (float)(z * s1 + w * c1));
}

__device__ __forceinline__ uint32_t e4m3x4(float4 v) {
    uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v.x, v.y), __NV_SATFINITE, __NV_E4M3);
    uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v.z, v.w), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// kRatio 2: the 2:1 layers (pairs pooled); kRatio 1: the 1:1 layers, where
// pooling is skipped and raw token p is written as compressed row p.
template <int kRatio, bool kNvfp4, bool kWinE4M3>
__global__ void __launch_bounds__(kThreads)
k_compress_append(int n_new, const float* __restrict__ kv_new, const float* __restrict__ gate_new,
                  float* pend_kv, float* pend_gate, void* const* comp,
                  uint8_t* const* comp_scales, const int64_t* comp_cap, void* const* win,
                  int32_t* n_tokens, int advance_here, RopeArgs rope, int32_t* dev_status) {
    const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    trace_start(kTraceCompress);
    // A kernel launched programmatically behind this one (the next append, the
    // Indexer) may be placed now; it waits for this grid before touching its data.
    // This one is launched the same way: nothing is read or written before the
    // kernels ahead of it on the stream have completed.
    sm100::grid_dep_launch_dependents();
    sm100::grid_dep_wait();
    const int ch = 4 * tid;
    const int64_t T = n_tokens[b];
    if (T < 0) {
        if (tid == 0 && c == 0) raise_status(dev_status, CSA2_DEV_BAD_LENGTH);
        return;
    }
    const float* kvb = kv_new + (int64_t)b * n_new * kD;
    const float* gb = gate_new ? gate_new + (int64_t)b * n_new * kD : nullptr;
    float* pk = pend_kv ? pend_kv + (int64_t)b * kD : nullptr;
    float* pg = pend_gate ? pend_gate + (int64_t)b * kD : nullptr;
    const bool has_comp = comp != nullptr;

    if (has_comp) {
        const int64_t cap = comp_cap[b];
        // rows completed by this call: pairs (2j, 2j+1) with j in [T/2, (T+n_new)/2),
        // or (ratio 1) the raw tokens j in [T, T+n_new)
        const int64_t j_lo = kRatio == 2 ? T >> 1 : T;
        const int64_t j_hi = kRatio == 2 ? (T + n_new) >> 1 : T + n_new;
        const int64_t j0 = j_lo + (int64_t)c * kPairsPerCta;
        const int64_t j1 = min(j_hi, j0 + kPairsPerCta);
        for (int64_t j = j0; j < j1; ++j) {
            float4 v;
            if constexpr (kRatio == 1) {
                v = ld4(kvb + (j - T) * kD + ch);
            } else {
                const int64_t t0 = 2 * j - T, t1 = t0 + 1;  // rows of kv_new; t0 = -1: pending
                float4 k0, g0;
                if (t0 < 0) {
                    k0 = ld4(pk + ch);
                    g0 = ld4(pg + ch);
                } else {
                    k0 = ld4(kvb + t0 * kD + ch);
                    g0 = ld4(gb + t0 * kD + ch);
                }
                const float4 k1 = ld4(kvb + t1 * kD + ch), g1 = ld4(gb + t1 * kD + ch);
                v.x = pool1(k0.x, k1.x, g0.x, g1.x);
                v.y = pool1(k0.y, k1.y, g0.y, g1.y);
                v.z = pool1(k0.z, k1.z, g0.z, g1.z);
                v.w = pool1(k0.w, k1.w, g0.w, g1.w);
            }
            v = rope4(v, ch, (int64_t)kRatio * j, rope);  // row j sits at raw position ratio*j
            if (j >= cap) {
                if (tid == 0) raise_status(dev_status, CSA2_DEV_BAD_LENGTH);
                continue;
            }
            if constexpr (kNvfp4) {
                uint8_t sb;
                const uint32_t codes = nvfp4_4(v, sb);
                uint8_t* vals = static_cast<uint8_t*>(comp[b]) + j * (kD / 2);
                *reinterpret_cast<uint16_t*>(vals + 2 * tid) = (uint16_t)codes;
                if ((tid & 3) == 0) comp_scales[b][j * (kD / kGroup) + (tid >> 2)] = sb;
            } else {
                st4(static_cast<float*>(comp[b]) + j * kD + ch, v);
            }
        }
    }

    // ring window: only the newest W of the new tokens survive, spread over CTAs
    for (int i = max(0, n_new - kW) + c; i < n_new; i += gridDim.x) {
        const int slot = (int)((T + i) % kW);
        const float4 k = ld4(kvb + (int64_t)i * kD + ch);
        if constexpr (kWinE4M3)
            *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(win[b]) + slot * kD + ch) = e4m3x4(k);
        else
            st4(static_cast<float*>(win[b]) + slot * kD + ch, k);
    }

    if (kRatio == 2 && has_comp && c == 0 && ((T + n_new) & 1) && n_new > 0) {
        // the last token starts a pair that completes later. The pending read
        // above (pair T/2 when T is odd) happened in this CTA, same channels.
        __syncthreads();
        st4(pk + ch, ld4(kvb + (int64_t)(n_new - 1) * kD + ch));
        st4(pg + ch, ld4(gb + (int64_t)(n_new - 1) * kD + ch));
    }
    if (advance_here) {
        __syncthreads();
        if (tid == 0) n_tokens[b] = (int32_t)(T + n_new);
    }
    trace_end(kTraceCompress);
}

__global__ void k_advance(int32_t* n_tokens, int B, int n_new) {
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B && n_tokens[b] >= 0) n_tokens[b] += n_new;
}

// Standalone quantiser: 4 elements per thread, 4 lanes per 16-element group.
__global__ void __launch_bounds__(256)
k_nvfp4_quantize(const float* __restrict__ x, int64_t n_elems, uint8_t* vals, uint8_t* scales) {
    const int64_t e = 4 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x);
    const bool live = e < n_elems;
    const float4 v = live ? ld4(x + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    uint8_t sb;
    const uint32_t codes = nvfp4_4(v, sb);
    if (!live) return;
    *reinterpret_cast<uint16_t*>(vals + e / 2) = (uint16_t)codes;
    if (((e >> 2) & 3) == 0) scales[e / kGroup] = sb;
}

// Linear prefill window: rows i < W-1 copy raw position T-(W-1)+i from the
// ring (zero when negative), rows W-1+t cast chunk token t to E4M3.
__global__ void __launch_bounds__(kThreads)
k_window_linear(int n_new, const float* __restrict__ kv_new, const void* const* win,
                const int32_t* __restrict__ n_tokens, uint8_t* out) {
    const int b = blockIdx.y, tid = threadIdx.x, ch = 4 * tid;
    const int rows = kW - 1 + n_new;
    const int64_t T = n_tokens[b];
    for (int i = blockIdx.x; i < rows; i += gridDim.x) {
        uint32_t v;
        if (i < kW - 1) {
            const int64_t pos = T - (kW - 1) + i;
            v = pos < 0 ? 0u
                        : *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(win[b]) +
                                                             (pos % kW) * kD + ch);
        } else {
            v = e4m3x4(ld4(kv_new + ((int64_t)b * n_new + (i - (kW - 1))) * kD + ch));
        }
        *reinterpret_cast<uint32_t*>(out + ((int64_t)b * rows + i) * kD + ch) = v;
    }
}

}  // namespace

CSA2_TRACE_SETTER(trace_set_compress)

cudaError_t preload_compress() {
    cudaError_t (*l[])() = {
        [] { return preload_kernel(k_compress_append<2, true, true>); },
        [] { return preload_kernel(k_compress_append<2, true, false>); },
        [] { return preload_kernel(k_compress_append<2, false, true>); },
        [] { return preload_kernel(k_compress_append<2, false, false>); },
        [] { return preload_kernel(k_compress_append<1, true, true>); },
        [] { return preload_kernel(k_compress_append<1, true, false>); },
        [] { return preload_kernel(k_compress_append<1, false, true>); },
        [] { return preload_kernel(k_compress_append<1, false, false>); },
        [] { return preload_kernel(k_advance); },
        [] { return preload_kernel(k_nvfp4_quantize); },
        [] { return preload_kernel(k_window_linear); }};
    for (auto f : l)
        if (const cudaError_t e = f()) return e;
    return cudaSuccess;
}

}  // namespace csa2

using namespace csa2;

extern "C" int csa2_window_linear(const csa2_params* p, int B, int n_new, const float* kv_new,
                                  const void* const* win, const int32_t* n_tokens, uint8_t* out,
                                  void* stream) {
    CSA2_CHECK_PARAMS(p);
    if (B < 0 || n_new < 0) return fail(CSA2_ERR_INVALID_ARG, "window_linear: negative size");
    if (B == 0) return CSA2_OK;
    if (p->head_dim != kD || p->window != kW || p->win_format != CSA2_E4M3)
        return fail(CSA2_ERR_UNSUPPORTED, "window_linear: built for D=512, W=128, E4M3 windows");
    if ((n_new && !kv_new) || !win || !n_tokens || !out)
        return fail(CSA2_ERR_INVALID_ARG, "window_linear: NULL buffer");
    if ((kv_new && !aligned16(kv_new)) || !aligned16(out))
        return fail(CSA2_ERR_ALIGN, "window_linear: kv_new and out must be 16-byte aligned");
    const int rows = kW - 1 + n_new;
    const int gx = rows < 1024 ? rows : 1024;
    if (const int rc = ensure_loaded()) return rc;
    k_window_linear<<<dim3(gx, B), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        n_new, kv_new, win, n_tokens, out);
    return check_launch("window_linear");
}

extern "C" int csa2_compress_append(const csa2_params* p, int B, int n_new,
                                    const float* kv_new, const float* gate_new,
                                    float* pend_kv, float* pend_gate,
                                    void* const* comp, uint8_t* const* comp_scales,
                                    const int64_t* comp_cap, void* const* win, int32_t* n_tokens,
                                    int32_t* dev_status, void* stream) {
    CSA2_CHECK_PARAMS(p);
    if (B < 0 || n_new < 0) return fail(CSA2_ERR_INVALID_ARG, "compress_append: negative size");
    if (B == 0 || n_new == 0) return CSA2_OK;
    if (p->head_dim != kD || p->window != kW || (p->compress_ratio != 2 && p->compress_ratio != 1))
        return fail(CSA2_ERR_UNSUPPORTED, "compress_append: built for D=512, W=128, ratio 2 or 1");
    const int ratio = p->compress_ratio;
    if (!kv_new || !win || !n_tokens)
        return fail(CSA2_ERR_INVALID_ARG, "compress_append: kv_new, win, n_tokens are required");
    if (comp && (!comp_cap || (ratio == 2 && (!gate_new || !pend_kv || !pend_gate))))
        return fail(CSA2_ERR_INVALID_ARG,
                    "compress_append: comp_cap (and at ratio 2 gate and pending state) required with comp");
    const bool nvfp4 = p->kv_format == CSA2_NVFP4;
    if (comp && !nvfp4 && p->kv_format != CSA2_F32)
        return fail(CSA2_ERR_UNSUPPORTED, "compress_append: kv_format must be NVFP4 or F32");
    if (comp && nvfp4 && !comp_scales)
        return fail(CSA2_ERR_INVALID_ARG, "compress_append: NVFP4 needs comp_scales");
    if (p->win_format != CSA2_E4M3 && p->win_format != CSA2_F32)
        return fail(CSA2_ERR_UNSUPPORTED, "compress_append: win_format must be E4M3 or F32");
    if (p->rope_dim < 0 || p->rope_dim > kD || p->rope_dim % 4)
        return fail(CSA2_ERR_UNSUPPORTED, "compress_append: rope_dim must be a multiple of 4 in [0, 512]");
    if (p->rope_dim > 0 && !(p->rope_theta > 0.f && p->rope_factor > 0.f && p->rope_orig_len > 0.f &&
                             p->rope_beta_fast > p->rope_beta_slow))
        return fail(CSA2_ERR_INVALID_ARG,
                    "compress_append: rope needs theta, factor, orig_len > 0 and beta_fast > beta_slow");
    RopeArgs rope;
    rope.dim = comp ? p->rope_dim : 0;
    rope.base = p->rope_theta;
    rope.factor = p->rope_factor;
    rope.orig_len = p->rope_orig_len;
    rope.beta_fast = p->rope_beta_fast;
    rope.beta_slow = p->rope_beta_slow;
    if (!aligned16(kv_new) || (gate_new && !aligned16(gate_new)) ||
        (pend_kv && !aligned16(pend_kv)) || (pend_gate && !aligned16(pend_gate)))
        return fail(CSA2_ERR_ALIGN, "compress_append: fp32 buffers must be 16-byte aligned");

    const int rows = ratio == 2 ? n_new / 2 + 1 : n_new;  // compressed rows this call can complete
    const int gx = comp ? (rows + kPairsPerCta - 1) / kPairsPerCta : 1;
    const int advance_here = gx == 1;
    const dim3 grid(gx, B);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool we = p->win_format == CSA2_E4M3;
    if (const int rc = ensure_loaded()) return rc;
    // programmatic launch: the CTAs may be placed while the kernel ahead still runs
    // (they wait for it first), which hides the launch gap between back-to-back appends
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#define CSA2_LAUNCH(R, NV, WE)                                                                       \
    do {                                                                                             \
        if (cudaLaunchKernelEx(&cfg, k_compress_append<R, NV, WE>, n_new, kv_new, gate_new, pend_kv, \
                               pend_gate, comp, comp_scales, comp_cap, win, n_tokens, advance_here,  \
                               rope, dev_status) != cudaSuccess)                                     \
            return check_launch("compress_append");                                                  \
    } while (0)
    if (ratio == 2) {
        if (nvfp4 && we) CSA2_LAUNCH(2, true, true);
        else if (nvfp4) CSA2_LAUNCH(2, true, false);
        else if (we) CSA2_LAUNCH(2, false, true);
        else CSA2_LAUNCH(2, false, false);
    } else {
        if (nvfp4 && we) CSA2_LAUNCH(1, true, true);
        else if (nvfp4) CSA2_LAUNCH(1, true, false);
        else if (we) CSA2_LAUNCH(1, false, true);
        else CSA2_LAUNCH(1, false, false);
    }
#undef CSA2_LAUNCH
    if (!advance_here) k_advance<<<(B + 127) / 128, 128, 0, s>>>(n_tokens, B, n_new);
    return check_launch("compress_append");
}

extern "C" int csa2_nvfp4_quantize(const float* x, int64_t n_rows, int row_len, uint8_t* vals,
                                   uint8_t* scales, void* stream) {
    if (n_rows < 0 || row_len <= 0 || row_len % kGroup)
        return fail(CSA2_ERR_SHAPE, "nvfp4_quantize: row_len must be a positive multiple of 16");
    if (n_rows == 0) return CSA2_OK;
    if (!x || !vals || !scales) return fail(CSA2_ERR_INVALID_ARG, "nvfp4_quantize: NULL buffer");
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(vals) & 1))
        return fail(CSA2_ERR_ALIGN, "nvfp4_quantize: x 16-byte, vals 2-byte aligned");
    const int64_t n = n_rows * (int64_t)row_len;
    const int64_t threads = n / 4;
    const int64_t blocks = (threads + 255) / 256;
    if (const int rc = ensure_loaded()) return rc;
    k_nvfp4_quantize<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, n, vals,
                                                                                      scales);
    return check_launch("nvfp4_quantize");
}
