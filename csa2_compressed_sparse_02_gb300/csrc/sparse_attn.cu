// Sparse attention over the 128-slot window plus the selected compressed
// positions, with a per-head sink logit in the softmax denominator.
// "DeepSeek-V4.1-Flash-NVFP4" §3.4 (gather by index, online softmax, built-in
// attn_sink, no n x n matrix), §三 (128 + 512 = 640 positions per query), §3.1
// (FP8 window), §一 (one 512-d KV head shared by the query heads, MLA style,
// so K = V = the latent).
//
// Split-KV: the 640 positions are 5 chunks of 128 (chunk 0 = window ring,
// chunks 1..4 = idx[0..512) in 128s). One CTA per (chunk, sequence) computes
// the chunk's unnormalised P.V, row max and row sum for all 64 heads; a merge
// kernel combines the 5 chunks and the sink with a log-sum-exp. Logits live in
// the log2 domain (scaled by log2 e) so that exp2 is the only transcendental.
//
// bf16 path: the gathered rows are decoded exactly into bf16 in shared memory
// (E2M1 x E4M3 has <= 6 significant bits, E4M3 has 4) and both products run on
// tensor cores with fp32 accumulation; P is rounded to bf16 and the row sums
// use the same rounded P, so the weights stay consistent.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kSplits = 5;
constexpr int kRows = 128;         // positions per split
constexpr int kThreads = 256;      // 8 warps
constexpr float kLog2e = 1.4426950408889634f;

// ---- shared memory layout of the bf16 kernel (bytes) ----
constexpr int kQBytes = kH * kD * 2;        // 64 KB, rows of 1024 B
constexpr int kKVBytes = kRows * kD * 2;    // 128 KB
constexpr int kPBytes = kH * kRows * 2;     // 16 KB, rows of 256 B
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQBytes;
constexpr int kOffP = kOffKV + kKVBytes;
constexpr int kOffRed = kOffP + kPBytes;    // float red_max[2][64], red_sum[2][64]
constexpr int kOffValid = kOffRed + 4 * kH * 4;
constexpr int kSmemBf16 = kOffValid + kRows * 4;

// 16-byte chunk c of row r of a tile whose rows hold `chunks` 16-byte chunks,
// XOR-swizzled on the low 3 bits so ldmatrix row groups hit distinct banks.
__device__ __forceinline__ uint32_t swz(int r, int c, int chunks) {
    return (uint32_t)((r * chunks + (c ^ (r & 7))) * 16);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h2) {
    return make_float2(__half2float(__ushort_as_half((uint16_t)(h2 & 0xffff))),
                       __half2float(__ushort_as_half((uint16_t)(h2 >> 16))));
}

// 8 E2M1 bytes (16 elements, element 0 = low nibble of byte 0) times scale s -> 8 bf16x2
__device__ __forceinline__ void nvfp4x16_to_bf16(uint2 v, float s, uint32_t* o) {
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 f = half2_bits_to_float2(e2m1x2_to_half2((w[i / 4] >> (8 * (i % 4))) & 0xffu));
        o[i] = pack_bf16(f.x * s, f.y * s);
    }
}

// 16 E4M3 bytes -> 8 bf16x2 (exact)
__device__ __forceinline__ void e4m3x16_to_bf16(uint4 v, uint32_t* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint16_t two = (uint16_t)((w[i / 2] >> (16 * (i % 2))) & 0xffffu);
        __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
        const float2 f = __half22float2(__half2(h));
        o[i] = pack_bf16(f.x, f.y);
    }
}

// Valid window row r for a sequence of T raw tokens. Ring layout: the ring
// holds raw positions max(0,T-W)..T-1, position p in slot p mod W. Linear
// layout: row r holds raw position T-W+r.
__device__ __forceinline__ bool window_slot_valid(int r, int64_t T, int linear) {
    return linear ? T - kW + r >= 0 : (T >= kW || (int64_t)r < T);
}

__global__ void __launch_bounds__(kThreads, 1)
k_sparse_attn_bf16(const __nv_bfloat16* __restrict__ q, const void* const* win,
                   const int32_t* __restrict__ n_tokens, const void* const* comp,
                   const uint8_t* const* comp_scales, const int32_t* __restrict__ idx, int ratio,
                   float scale_log2, float* ws_o, float2* ws_ml, int32_t* dev_status,
                   int win_linear) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int split = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char* sQ = smem + kOffQ;
    unsigned char* sKV = smem + kOffKV;
    unsigned char* sP = smem + kOffP;
    float* red_max = reinterpret_cast<float*>(smem + kOffRed);  // [2][64]
    float* red_sum = red_max + 2 * kH;                           // [2][64]
    int* sValid = reinterpret_cast<int*>(smem + kOffValid);
    const int64_t T = n_tokens[b];
    const int64_t n_c = T / ratio;

    // ---- Q -> shared (async 16-byte copies) ----
    const unsigned char* qb = reinterpret_cast<const unsigned char*>(q + (int64_t)b * kH * kD);
#pragma unroll 4
    for (int e = tid; e < kH * (kD / 8); e += kThreads) {
        const int r = e / (kD / 8), c = e % (kD / 8);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(sQ + swz(r, c, 64))),
                     "l"(qb + (int64_t)e * 16));
    }
    asm volatile("cp.async.commit_group;\n");

    // ---- gather + exact decode of this split's 128 rows -> bf16 shared ----
    int any_valid = 0;
    for (int r = warp; r < kRows; r += kThreads / 32) {
        uint32_t o[8];
        bool valid;
        if (split == 0) {
            valid = T > 0 && window_slot_valid(r, T, win_linear);
            if (valid) {
                const uint4 v = *reinterpret_cast<const uint4*>(
                    static_cast<const uint8_t*>(win[b]) + (int64_t)r * kD + 16 * lane);
                e4m3x16_to_bf16(v, o);
            }
        } else {
            const int64_t j = idx[(int64_t)b * kKp + (split - 1) * kRows + r];
            valid = j >= 0 && j < n_c;
            if (j >= n_c && lane == 0) raise_status(dev_status, CSA2_DEV_BAD_INDEX);
            if (valid) {
                const uint2 v = *reinterpret_cast<const uint2*>(
                    static_cast<const uint8_t*>(comp[b]) + j * (kD / 2) + 8 * lane);
                const float s = e4m3_value(comp_scales[b][j * (kD / kGroup) + lane]);
                nvfp4x16_to_bf16(v, s, o);
            }
        }
        if (!valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = 0u;
        }
        *reinterpret_cast<uint4*>(sKV + swz(r, 2 * lane, 64)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(sKV + swz(r, 2 * lane + 1, 64)) = make_uint4(o[4], o[5], o[6], o[7]);
        if (lane == 0) sValid[r] = valid;
        any_valid |= valid;
    }
    asm volatile("cp.async.wait_all;\n");
    if (!__syncthreads_or(any_valid)) {  // nothing to attend in this split
        if (tid < kH) ws_ml[((int64_t)b * kSplits + split) * kH + tid] = make_float2(-INFINITY, 0.f);
        return;
    }

    // ---- S = Q K^T : warp -> rows 16*(warp&3), columns 64*(warp>>2) ----
    const int m0 = 16 * (warp & 3), n0 = 64 * (warp >> 2);
    const int g = lane >> 2, t = lane & 3;
    float s_acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s_acc[j][0] = s_acc[j][1] = s_acc[j][2] = s_acc[j][3] = 0.f;
    const uint32_t sQ_u = smem_u32(sQ), sKV_u = smem_u32(sKV), sP_u = smem_u32(sP);
#pragma unroll 2
    for (int kk = 0; kk < kD / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sQ_u + swz(m0 + (lane & 15), 2 * kk + (lane >> 4), 64), a0, a1, a2, a3);
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
            uint32_t b0, b1, b2, b3;
            const int nrow = n0 + 16 * jp + (lane & 7) + ((lane >> 4) << 3);
            ldsm_x4(sKV_u + swz(nrow, 2 * kk + ((lane >> 3) & 1), 64), b0, b1, b2, b3);
            mma_bf16(s_acc[2 * jp], a0, a1, a2, a3, b0, b1);
            mma_bf16(s_acc[2 * jp + 1], a0, a1, a2, a3, b2, b3);
        }
    }

    // ---- chunk softmax statistics (log2 domain) ----
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int c0 = n0 + 8 * j + 2 * t;
        const bool v0 = sValid[c0], v1 = sValid[c0 + 1];
        s_acc[j][0] = v0 ? s_acc[j][0] * scale_log2 : -INFINITY;
        s_acc[j][1] = v1 ? s_acc[j][1] * scale_log2 : -INFINITY;
        s_acc[j][2] = v0 ? s_acc[j][2] * scale_log2 : -INFINITY;
        s_acc[j][3] = v1 ? s_acc[j][3] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(s_acc[j][0], s_acc[j][1]));
        mx1 = fmaxf(mx1, fmaxf(s_acc[j][2], s_acc[j][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (t == 0) {
        red_max[(warp >> 2) * kH + m0 + g] = mx0;
        red_max[(warp >> 2) * kH + m0 + g + 8] = mx1;
    }
    __syncthreads();
    float rm0 = fmaxf(red_max[m0 + g], red_max[kH + m0 + g]);
    float rm1 = fmaxf(red_max[m0 + g + 8], red_max[kH + m0 + g + 8]);
    const float base0 = rm0 == -INFINITY ? 0.f : rm0;
    const float base1 = rm1 == -INFINITY ? 0.f : rm1;
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const __nv_bfloat162 p01 = __floats2bfloat162_rn(exp2f(s_acc[j][0] - base0),
                                                         exp2f(s_acc[j][1] - base0));
        const __nv_bfloat162 p23 = __floats2bfloat162_rn(exp2f(s_acc[j][2] - base1),
                                                         exp2f(s_acc[j][3] - base1));
        const float2 f01 = __bfloat1622float2(p01), f23 = __bfloat1622float2(p23);
        sum0 += f01.x + f01.y;
        sum1 += f23.x + f23.y;
        const int col = n0 + 8 * j + 2 * t;  // element column; chunk = col/8, byte = (col%8)*2
        *reinterpret_cast<__nv_bfloat162*>(sP + swz(m0 + g, col >> 3, 16) + (col & 7) * 2) = p01;
        *reinterpret_cast<__nv_bfloat162*>(sP + swz(m0 + g + 8, col >> 3, 16) + (col & 7) * 2) = p23;
    }
    sum0 += __shfl_xor_sync(0xffffffffu, sum0, 1);
    sum0 += __shfl_xor_sync(0xffffffffu, sum0, 2);
    sum1 += __shfl_xor_sync(0xffffffffu, sum1, 1);
    sum1 += __shfl_xor_sync(0xffffffffu, sum1, 2);
    if (t == 0) {
        red_sum[(warp >> 2) * kH + m0 + g] = sum0;
        red_sum[(warp >> 2) * kH + m0 + g + 8] = sum1;
    }
    __syncthreads();
    if (warp < 4 && t == 0) {
        float2* ml = ws_ml + ((int64_t)b * kSplits + split) * kH;
        ml[m0 + g] = make_float2(rm0, red_sum[m0 + g] + red_sum[kH + m0 + g]);
        ml[m0 + g + 8] = make_float2(rm1, red_sum[m0 + g + 8] + red_sum[kH + m0 + g + 8]);
    }

    // ---- O = P V : warp -> rows m0, columns 256*(warp>>2) in two halves of 128 ----
    float* ob = ws_o + ((int64_t)b * kSplits + split) * kH * kD;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        const int c0 = 256 * (warp >> 2) + 128 * half;
        float o_acc[16][4];
#pragma unroll
        for (int j = 0; j < 16; ++j) o_acc[j][0] = o_acc[j][1] = o_acc[j][2] = o_acc[j][3] = 0.f;
#pragma unroll 2
        for (int kk = 0; kk < kRows / 16; ++kk) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sP_u + swz(m0 + (lane & 15), 2 * kk + (lane >> 4), 16), a0, a1, a2, a3);
#pragma unroll
            for (int jp = 0; jp < 8; ++jp) {
                uint32_t b0, b1, b2, b3;
                const int prow = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
                ldsm_x4_t(sKV_u + swz(prow, (c0 >> 3) + 2 * jp + (lane >> 4), 64), b0, b1, b2, b3);
                mma_bf16(o_acc[2 * jp], a0, a1, a2, a3, b0, b1);
                mma_bf16(o_acc[2 * jp + 1], a0, a1, a2, a3, b2, b3);
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int col = c0 + 8 * j + 2 * t;
            *reinterpret_cast<float2*>(ob + (int64_t)(m0 + g) * kD + col) =
                make_float2(o_acc[j][0], o_acc[j][1]);
            *reinterpret_cast<float2*>(ob + (int64_t)(m0 + g + 8) * kD + col) =
                make_float2(o_acc[j][2], o_acc[j][3]);
        }
    }
}

// ---- fp32 (unquantised) path, CUDA cores: one thread per row for Q.K, one
// thread per 4 output channels for P.V ----
constexpr int kF32Threads = 128;
constexpr int kSmemF32 = (kD * kH + kH * kRows) * 4;

__global__ void __launch_bounds__(kF32Threads)
k_sparse_attn_f32(const float* __restrict__ q, const void* const* win,
                  const int32_t* __restrict__ n_tokens, const void* const* comp,
                  const int32_t* __restrict__ idx, int ratio, float scale_log2, float* ws_o,
                  float2* ws_ml, int32_t* dev_status, int win_linear) {
    extern __shared__ __align__(1024) unsigned char smem[];
    float* sQt = reinterpret_cast<float*>(smem);  // [D][H]
    float* sS = sQt + kD * kH;                     // [H][rows]
    __shared__ const float* sRow[kRows];
    const int split = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int64_t T = n_tokens[b], n_c = T / ratio;
    for (int e = tid; e < kH * kD; e += kF32Threads) {
        const int h = e / kD, d = e % kD;
        sQt[d * kH + h] = q[(int64_t)b * kH * kD + e];
    }
    {
        const int r = tid;
        const float* row = nullptr;
        if (split == 0) {
            if (T > 0 && window_slot_valid(r, T, win_linear))
                row = static_cast<const float*>(win[b]) + (int64_t)r * kD;
        } else {
            const int64_t j = idx[(int64_t)b * kKp + (split - 1) * kRows + r];
            if (j >= n_c) raise_status(dev_status, CSA2_DEV_BAD_INDEX);
            if (j >= 0 && j < n_c) row = static_cast<const float*>(comp[b]) + j * kD;
        }
        sRow[r] = row;
    }
    __syncthreads();
    {
        const int r = tid;
        const float* row = sRow[r];
        float acc[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) acc[h] = 0.f;
        if (row) {
            for (int d = 0; d < kD; d += 4) {
                const float4 k = *reinterpret_cast<const float4*>(row + d);
                const float kv[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4* qd = reinterpret_cast<const float4*>(sQt + (d + i) * kH);
#pragma unroll
                    for (int h4 = 0; h4 < kH / 4; ++h4) {
                        const float4 a = qd[h4];
                        acc[4 * h4 + 0] = fmaf(a.x, kv[i], acc[4 * h4 + 0]);
                        acc[4 * h4 + 1] = fmaf(a.y, kv[i], acc[4 * h4 + 1]);
                        acc[4 * h4 + 2] = fmaf(a.z, kv[i], acc[4 * h4 + 2]);
                        acc[4 * h4 + 3] = fmaf(a.w, kv[i], acc[4 * h4 + 3]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < kH; ++h) sS[h * kRows + r] = row ? acc[h] * scale_log2 : -INFINITY;
    }
    __syncthreads();
    if (tid < kH) {
        const int h = tid;
        float m = -INFINITY;
        for (int r = 0; r < kRows; ++r) m = fmaxf(m, sS[h * kRows + r]);
        const float base = m == -INFINITY ? 0.f : m;
        float l = 0.f;
        for (int r = 0; r < kRows; ++r) {
            const float p = exp2f(sS[h * kRows + r] - base);
            sS[h * kRows + r] = p;
            l += p;
        }
        ws_ml[((int64_t)b * kSplits + split) * kH + h] = make_float2(m, l);
    }
    __syncthreads();
    float* ob = ws_o + ((int64_t)b * kSplits + split) * kH * kD;
    const int d = 4 * tid;
    for (int h0 = 0; h0 < kH; h0 += 16) {
        float4 acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < kRows; ++r) {
            const float* row = sRow[r];
            if (!row) continue;
            const float4 v = *reinterpret_cast<const float4*>(row + d);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float p = sS[(h0 + i) * kRows + r];
                acc[i].x = fmaf(p, v.x, acc[i].x);
                acc[i].y = fmaf(p, v.y, acc[i].y);
                acc[i].z = fmaf(p, v.z, acc[i].z);
                acc[i].w = fmaf(p, v.w, acc[i].w);
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) *reinterpret_cast<float4*>(ob + (int64_t)(h0 + i) * kD + d) = acc[i];
    }
}

// ---- merge of the 5 split results and the sink: one CTA per (head, sequence) ----
template <bool kBf16Out>
__global__ void __launch_bounds__(128)
k_sparse_attn_merge(const float* __restrict__ sink, const float* __restrict__ ws_o,
                    const float2* __restrict__ ws_ml, void* out) {
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const float sink2 = sink[h] * kLog2e;
    float2 ml[kSplits];
    float M = sink2;
#pragma unroll
    for (int s = 0; s < kSplits; ++s) {
        ml[s] = ws_ml[((int64_t)b * kSplits + s) * kH + h];
        if (ml[s].y > 0.f) M = fmaxf(M, ml[s].x);
    }
    float L = exp2f(sink2 - M), wgt[kSplits];
#pragma unroll
    for (int s = 0; s < kSplits; ++s) {
        wgt[s] = ml[s].y > 0.f ? exp2f(ml[s].x - M) : 0.f;
        L += ml[s].y * wgt[s];
    }
    const float inv = 1.0f / L;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kSplits; ++s) {
        if (wgt[s] == 0.f) continue;
        const float4 o = *reinterpret_cast<const float4*>(
            ws_o + (((int64_t)b * kSplits + s) * kH + h) * kD + 4 * tid);
        acc.x = fmaf(wgt[s], o.x, acc.x);
        acc.y = fmaf(wgt[s], o.y, acc.y);
        acc.z = fmaf(wgt[s], o.z, acc.z);
        acc.w = fmaf(wgt[s], o.w, acc.w);
    }
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    const int64_t off = ((int64_t)b * kH + h) * kD + 4 * tid;
    if constexpr (kBf16Out) {
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + off) =
            make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + off) = acc;
    }
}

// ---- fused multi-layer flash-decode (bf16 tensor cores, output in registers) ----
// One CTA per (layer, sequence): 64 query heads x all 640 positions, streamed
// as 10 chunks of 64 positions (2 window chunks, 8 compressed chunks) with an
// online softmax. The output O[64 x 512] lives in registers: warp w owns all
// 64 rows and dims 32w..32w+31 (4 x 4 mma tiles, 64 fp32 per thread), so each
// V fragment is read from shared memory once per chunk. The
// next chunk's raw bytes are loaded into registers while the current chunk is
// multiplied, then decoded exactly into bf16 shared memory. The sink joins the
// denominator once at the end; no workspace, no merge pass. All L layers of a
// launch share the compressed cache and the selected indices.
constexpr int kFdWarps = 16;
constexpr int kFdThreads = 32 * kFdWarps;
constexpr int kFdChunk = 64;
constexpr int kFdChunks = (kW + kKp) / kFdChunk;  // 10
constexpr int kFdOffQ = 0;                                  // 64 x 1024 B
constexpr int kFdOffKV = kFdOffQ + kH * kD * 2;             // 2 x 64 x 1024 B
constexpr int kFdOffP = kFdOffKV + 2 * kFdChunk * kD * 2;    // 64 x 128 B
constexpr int kFdOffMax = kFdOffP + kH * kFdChunk * 2;       // float [5][64]: maxima, alpha
constexpr int kFdOffSum = kFdOffMax + 5 * kH * 4;            // float [4][64]
constexpr int kFdOffValid = kFdOffSum + 4 * kH * 4;          // int [2][64]
constexpr int kFdOffIdx = kFdOffValid + 2 * kFdChunk * 4;     // int [512] selected positions
constexpr int kSmemFd = kFdOffIdx + kKp * 4;

// Raw bytes of 4 rows of a chunk, per lane (the warp covers one row per step).
struct FdRaw {
    uint4 v[4];       // window: 16 E4M3 bytes; compressed: .x/.y = 8 E2M1 bytes
    uint32_t sc;      // compressed: the lane's group-scale byte, 4 rows packed
    uint32_t valid;   // bit r: row r of the 4 is valid
};

__device__ __forceinline__ void fd_load(FdRaw& raw, int c, int warp, int lane, int64_t T,
                                        int64_t n_c, const uint8_t* win, const uint8_t* comp,
                                        const uint8_t* comp_sc, const int32_t* idx,
                                        int32_t* dev_status, int win_linear) {
    raw.valid = 0;
    raw.sc = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = warp * 4 + k;  // row within the chunk
        raw.v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (c < kW / kFdChunk) {  // window chunk: ring slot c*64 + r
            const int slot = c * kFdChunk + r;
            if (T > 0 && window_slot_valid(slot, T, win_linear)) {
                raw.v[k] = *reinterpret_cast<const uint4*>(win + (int64_t)slot * kD + 16 * lane);
                raw.valid |= 1u << k;
            }
        } else {
            const int64_t j = idx[(c - kW / kFdChunk) * kFdChunk + r];
            if (j >= n_c && lane == 0) raise_status(dev_status, CSA2_DEV_BAD_INDEX);
            if (j >= 0 && j < n_c) {
                const uint2 v = *reinterpret_cast<const uint2*>(comp + j * (kD / 2) + 8 * lane);
                raw.v[k] = make_uint4(v.x, v.y, 0u, 0u);
                raw.sc |= (uint32_t)comp_sc[j * (kD / kGroup) + lane] << (8 * k);
                raw.valid |= 1u << k;
            }
        }
    }
}

__device__ __forceinline__ void fd_store(const FdRaw& raw, int c, int warp, int lane,
                                         unsigned char* sKV, int* sValid) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = warp * 4 + k;
        uint32_t o[8];
        const bool valid = (raw.valid >> k) & 1u;
        if (valid && c < kW / kFdChunk) {
            e4m3x16_to_bf16(raw.v[k], o);
        } else if (valid) {
            nvfp4x16_to_bf16(make_uint2(raw.v[k].x, raw.v[k].y),
                             e4m3_value((uint8_t)(raw.sc >> (8 * k))), o);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = 0u;
        }
        if (c < kW / kFdChunk) {  // window row: lane covers dims 16*lane..+15 = chunks 2l, 2l+1
            *reinterpret_cast<uint4*>(sKV + swz(r, 2 * lane, 64)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(sKV + swz(r, 2 * lane + 1, 64)) = make_uint4(o[4], o[5], o[6], o[7]);
        } else {  // compressed row: lane covers its 16-element group = dims 16*lane..+15
            *reinterpret_cast<uint4*>(sKV + swz(r, 2 * lane, 64)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(sKV + swz(r, 2 * lane + 1, 64)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        if (lane == 0) sValid[r] = valid;
    }
}

__global__ void __launch_bounds__(kFdThreads, 1)
k_sparse_attn_fd(int B, const __nv_bfloat16* __restrict__ q, const float* __restrict__ sink,
                 const void* const* win, const int32_t* __restrict__ n_tokens,
                 const void* const* comp, const uint8_t* const* comp_scales,
                 const int32_t* __restrict__ idx, int ratio, float scale_log2,
                 __nv_bfloat16* out, int32_t* dev_status, int win_linear) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int layer = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp & 3, wn = warp >> 2;  // row group (16 heads), column group
    const int g = lane >> 2, t = lane & 3;
    unsigned char* sQ = smem + kFdOffQ;
    unsigned char* sP = smem + kFdOffP;
    float* sMax = reinterpret_cast<float*>(smem + kFdOffMax);
    float* sSum = reinterpret_cast<float*>(smem + kFdOffSum);
    int* sValid = reinterpret_cast<int*>(smem + kFdOffValid);
    const int64_t T = n_tokens[b];
    const int64_t n_c = T / ratio;
    const int64_t lb = (int64_t)layer * B + b;
    const uint8_t* winb = static_cast<const uint8_t*>(win[lb]);
    const uint8_t* compb = static_cast<const uint8_t*>(comp[b]);
    const uint8_t* compsb = comp_scales[b];
    int32_t* sIdx = reinterpret_cast<int32_t*>(smem + kFdOffIdx);
    for (int i = tid; i < kKp; i += kFdThreads) sIdx[i] = idx[(int64_t)b * kKp + i];
    __syncthreads();
    const int32_t* idxb = sIdx;  // gathers read the indices from shared memory

    // ---- Q -> shared (async), chunk 0 -> shared ----
    const unsigned char* qb = reinterpret_cast<const unsigned char*>(q + lb * kH * kD);
    for (int e = tid; e < kH * (kD / 8); e += kFdThreads) {
        const int r = e / (kD / 8), c = e % (kD / 8);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(sQ + swz(r, c, 64))),
                     "l"(qb + (int64_t)e * 16));
    }
    asm volatile("cp.async.commit_group;\n");
    FdRaw raw;
    fd_load(raw, 0, warp, lane, T, n_c, winb, compb, compsb, idxb, dev_status, win_linear);
    fd_store(raw, 0, warp, lane, smem + kFdOffKV, sValid);
    asm volatile("cp.async.wait_all;\n");

    // O accumulator: all 64 rows (4 m-tiles) x dims 32*warp .. +31 (4 n-tiles)
    float o_acc[4][4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) o_acc[mt][j][0] = o_acc[mt][j][1] = o_acc[mt][j][2] = o_acc[mt][j][3] = 0.f;
    // running max / sum of rows 16wm+g, +8 (the S-phase rows of this thread)
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float* sAlpha = sMax;  // per-row rescale factor of the chunk, reuses the max buffer
    const uint32_t sQ_u = smem_u32(sQ), sP_u = smem_u32(sP);

    for (int c = 0; c < kFdChunks; ++c) {
        __syncthreads();  // chunk c in sKV[c&1] and its sValid are complete
        unsigned char* sKV = smem + kFdOffKV + (c & 1) * (kFdChunk * kD * 2);
        const int* vld = sValid + (c & 1) * kFdChunk;
        const uint32_t sKV_u = smem_u32(sKV);
        if (c + 1 < kFdChunks)
            fd_load(raw, c + 1, warp, lane, T, n_c, winb, compb, compsb, idxb, dev_status,
                    win_linear);

        // ---- S = Q K^T for rows 16wm.., positions 16wn.. (2 n-tiles) ----
        float s_acc[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) s_acc[j][0] = s_acc[j][1] = s_acc[j][2] = s_acc[j][3] = 0.f;
#pragma unroll 4
        for (int kk = 0; kk < kD / 16; ++kk) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(sQ_u + swz(16 * wm + (lane & 15), 2 * kk + (lane >> 4), 64), a0, a1, a2, a3);
            ldsm_x4(sKV_u + swz(16 * wn + (lane & 7) + ((lane >> 4) << 3), 2 * kk + ((lane >> 3) & 1), 64),
                    b0, b1, b2, b3);
            mma_bf16(s_acc[0], a0, a1, a2, a3, b0, b1);
            mma_bf16(s_acc[1], a0, a1, a2, a3, b2, b3);
        }
        // ---- online softmax (log2 domain) ----
        float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = 16 * wn + 8 * j + 2 * t;
            const bool v0 = vld[col], v1 = vld[col + 1];
            s_acc[j][0] = v0 ? s_acc[j][0] * scale_log2 : -INFINITY;
            s_acc[j][1] = v1 ? s_acc[j][1] * scale_log2 : -INFINITY;
            s_acc[j][2] = v0 ? s_acc[j][2] * scale_log2 : -INFINITY;
            s_acc[j][3] = v1 ? s_acc[j][3] * scale_log2 : -INFINITY;
            cm0 = fmaxf(cm0, fmaxf(s_acc[j][0], s_acc[j][1]));
            cm1 = fmaxf(cm1, fmaxf(s_acc[j][2], s_acc[j][3]));
        }
        cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, 1));
        cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, 2));
        cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, 1));
        cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, 2));
        if (t == 0) {
            sMax[wn * kH + 16 * wm + g] = cm0;
            sMax[wn * kH + 16 * wm + g + 8] = cm1;
        }
        __syncthreads();
        float n0 = m0, n1 = m1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            n0 = fmaxf(n0, sMax[k * kH + 16 * wm + g]);
            n1 = fmaxf(n1, sMax[k * kH + 16 * wm + g + 8]);
        }
        const float al0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
        const float al1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
        const float base0 = n0 == -INFINITY ? 0.f : n0, base1 = n1 == -INFINITY ? 0.f : n1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __nv_bfloat162 p01 = __floats2bfloat162_rn(exp2f(s_acc[j][0] - base0),
                                                             exp2f(s_acc[j][1] - base0));
            const __nv_bfloat162 p23 = __floats2bfloat162_rn(exp2f(s_acc[j][2] - base1),
                                                             exp2f(s_acc[j][3] - base1));
            const float2 f01 = __bfloat1622float2(p01), f23 = __bfloat1622float2(p23);
            ps0 += f01.x + f01.y;
            ps1 += f23.x + f23.y;
            const int col = 16 * wn + 8 * j + 2 * t;
            *reinterpret_cast<__nv_bfloat162*>(sP + swz(16 * wm + g, col >> 3, 8) + (col & 7) * 2) = p01;
            *reinterpret_cast<__nv_bfloat162*>(sP + swz(16 * wm + g + 8, col >> 3, 8) + (col & 7) * 2) = p23;
        }
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
        if (t == 0) {
            sSum[wn * kH + 16 * wm + g] = ps0;
            sSum[wn * kH + 16 * wm + g + 8] = ps1;
        }
        __syncthreads();
        float cs0 = 0.f, cs1 = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            cs0 += sSum[k * kH + 16 * wm + g];
            cs1 += sSum[k * kH + 16 * wm + g + 8];
        }
        l0 = l0 * al0 + cs0;
        l1 = l1 * al1 + cs1;
        m0 = n0;
        m1 = n1;
        if (wn == 0 && t == 0) {  // publish the rescale factors of all 64 rows (slot 0)
            sAlpha[4 * kH + 16 * wm + g] = al0;
            sAlpha[4 * kH + 16 * wm + g + 8] = al1;
        }
        __syncthreads();
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const float a0 = sAlpha[4 * kH + 16 * mt + g], a1 = sAlpha[4 * kH + 16 * mt + g + 8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                o_acc[mt][j][0] *= a0;
                o_acc[mt][j][1] *= a0;
                o_acc[mt][j][2] *= a1;
                o_acc[mt][j][3] *= a1;
            }
        }
        // ---- O += P V: all 64 rows x dims 32*warp.. (4 n-tiles), 64 positions ----
#pragma unroll
        for (int kk = 0; kk < kFdChunk / 16; ++kk) {
            uint32_t bv[2][4];
#pragma unroll
            for (int jp = 0; jp < 2; ++jp) {
                const int prow = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
                ldsm_x4_t(sKV_u + swz(prow, 4 * warp + 2 * jp + (lane >> 4), 64), bv[jp][0], bv[jp][1],
                          bv[jp][2], bv[jp][3]);
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(sP_u + swz(16 * mt + (lane & 15), 2 * kk + (lane >> 4), 8), a0, a1, a2, a3);
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    mma_bf16(o_acc[mt][2 * jp], a0, a1, a2, a3, bv[jp][0], bv[jp][1]);
                    mma_bf16(o_acc[mt][2 * jp + 1], a0, a1, a2, a3, bv[jp][2], bv[jp][3]);
                }
            }
        }
        if (c + 1 < kFdChunks)
            fd_store(raw, c + 1, warp, lane, smem + kFdOffKV + ((c + 1) & 1) * (kFdChunk * kD * 2),
                     sValid + ((c + 1) & 1) * kFdChunk);
    }

    // ---- sink and normalisation, bf16 out ----
    __syncthreads();  // every warp is done reading the last chunk's rescale factors
    if (wn == 0 && t == 0) {  // final factor of every row: e^{m}/(e^{sink} + sum) in log2 form
        const float sink2 = sink[(int64_t)layer * kH + 16 * wm + g] * kLog2e;
        const float sink2b = sink[(int64_t)layer * kH + 16 * wm + g + 8] * kLog2e;
        const float M0 = fmaxf(m0, sink2), M1 = fmaxf(m1, sink2b);
        const float sc0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M0);
        const float sc1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M1);
        sAlpha[4 * kH + 16 * wm + g] = sc0 / (l0 * sc0 + exp2f(sink2 - M0));
        sAlpha[4 * kH + 16 * wm + g + 8] = sc1 / (l1 * sc1 + exp2f(sink2b - M1));
    }
    __syncthreads();
    __nv_bfloat16* ob = out + lb * kH * kD;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
        const float f0 = sAlpha[4 * kH + 16 * mt + g], f1 = sAlpha[4 * kH + 16 * mt + g + 8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = 32 * warp + 8 * j + 2 * t;
            *reinterpret_cast<uint32_t*>(ob + (int64_t)(16 * mt + g) * kD + col) =
                pack_bf16(o_acc[mt][j][0] * f0, o_acc[mt][j][1] * f0);
            *reinterpret_cast<uint32_t*>(ob + (int64_t)(16 * mt + g + 8) * kD + col) =
                pack_bf16(o_acc[mt][j][2] * f1, o_acc[mt][j][3] * f1);
        }
    }
}

size_t ws_o_bytes(int B) { return (size_t)B * kSplits * kH * kD * sizeof(float); }
size_t ws_ml_bytes(int B) { return (size_t)B * kSplits * kH * sizeof(float2); }

}  // namespace

cudaError_t preload_attn() {
    cudaError_t e = preload_kernel(k_sparse_attn_bf16, kSmemBf16);
    if (!e) e = preload_kernel(k_sparse_attn_f32, kSmemF32);
    if (!e) e = preload_kernel(k_sparse_attn_merge<true>);
    if (!e) e = preload_kernel(k_sparse_attn_merge<false>);
    if (!e) e = preload_kernel(k_sparse_attn_fd, kSmemFd);
    return e;
}

}  // namespace csa2

using namespace csa2;

extern "C" size_t csa2_sparse_attn_workspace_size(const csa2_params* p, int B) {
    if (B <= 0) return 0;
    // the larger of the two schedules' needs: the CUDA-core and mma.sync split-KV
    // passes (5 partials per sequence) and the tcgen05 kernel's cut units
    const size_t kv = ws_o_bytes(B) + ws_ml_bytes(B);
    const size_t tc = sparse_attn_tc_ws_bytes(p, B);
    return kv > tc ? kv : tc;
}

extern "C" int csa2_sparse_attn_layers_mma(const csa2_params* p, int L, int B, const void* q,
                                       const float* sink, const void* const* win,
                                       const int32_t* n_tokens, const void* const* comp,
                                       const uint8_t* const* comp_scales, const int32_t* idx,
                                       void* out, int32_t* dev_status, void* stream) {
    CSA2_CHECK_PARAMS(p);
    if (L < 0 || B < 0) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn_layers_mma: negative size");
    if (L == 0 || B == 0) return CSA2_OK;
    if (p->heads != kH || p->head_dim != kD || p->window != kW || p->topk_pos != kKp ||
        p->compress_ratio < 1)
        return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn_layers_mma: built for 64 heads x 512, W=128, k=512");
    if (p->kv_format != CSA2_NVFP4 || p->win_format != CSA2_E4M3 || p->q_format != CSA2_BF16)
        return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn_layers_mma: formats must be NVFP4, E4M3, BF16");
    if (!q || !sink || !win || !n_tokens || !comp || !comp_scales || !idx || !out)
        return fail(CSA2_ERR_INVALID_ARG, "sparse_attn_layers_mma: NULL buffer");
    if (!aligned16(q) || !aligned16(out))
        return fail(CSA2_ERR_ALIGN, "sparse_attn_layers_mma: q, out must be 16-byte aligned");
    if (L > 65535 || B > 65535) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn_layers_mma: grid too large");
    // loads the kernel and sets its shared-memory limit on this device, once per device
    if (const int rc = ensure_loaded()) return rc;
    k_sparse_attn_fd<<<dim3(L, B), kFdThreads, kSmemFd, static_cast<cudaStream_t>(stream)>>>(
        B, static_cast<const __nv_bfloat16*>(q), sink, win, n_tokens, comp, comp_scales, idx,
        p->compress_ratio, p->softmax_scale * kLog2e, static_cast<__nv_bfloat16*>(out), dev_status,
        p->win_layout == CSA2_WIN_LINEAR);
    return check_launch("sparse_attn_layers_mma");
}

namespace {
// Host checks shared by csa2_sparse_attn and csa2_sparse_attn_mma. Returns
// CSA2_OK with *quant set, -1 for an empty batch (nothing to do), or an error.
int check_single(const char* name, const csa2_params* p, int B, const void* q, const float* sink,
                 const void* const* win, const int32_t* n_tokens, const void* const* comp,
                 const uint8_t* const* comp_scales, const int32_t* idx, void* out, void* workspace,
                 size_t ws_bytes, bool* quant) {
    const std::string n(name);
    CSA2_CHECK_PARAMS(p);
    if (B < 0) return fail(CSA2_ERR_INVALID_ARG, n + ": negative batch");
    if (B == 0) return -1;
    if (p->heads != kH || p->head_dim != kD || p->window != kW || p->topk_pos != kKp ||
        p->compress_ratio < 1)
        return fail(CSA2_ERR_UNSUPPORTED, n + ": built for 64 heads x 512, W=128, k=512");
    if (!q || !sink || !win || !n_tokens || !comp || !idx || !out || !workspace)
        return fail(CSA2_ERR_INVALID_ARG, n + ": NULL buffer");
    if (ws_bytes < csa2_sparse_attn_workspace_size(p, B))
        return fail(CSA2_ERR_SHAPE, n + ": workspace smaller than the size query");
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace))
        return fail(CSA2_ERR_ALIGN, n + ": q, out, workspace must be 16-byte aligned");
    *quant = p->kv_format == CSA2_NVFP4 && p->win_format == CSA2_E4M3 && p->q_format == CSA2_BF16;
    const bool plain = p->kv_format == CSA2_F32 && p->win_format == CSA2_F32 &&
                       p->q_format == CSA2_F32;
    if (!*quant && !plain)
        return fail(CSA2_ERR_UNSUPPORTED,
                    n + ": formats must be (NVFP4, E4M3, BF16) or (F32, F32, F32)");
    if (*quant && !comp_scales) return fail(CSA2_ERR_INVALID_ARG, n + ": NVFP4 needs scales");
    return CSA2_OK;
}

// The split-KV passes (5 position splits per sequence, partials in the
// workspace) and the log-sum-exp merge: fp32 on CUDA cores, or bf16 mma.sync.
int launch_split_kv(const char* name, const csa2_params* p, int B, bool quant, const void* q,
                    const float* sink, const void* const* win, const int32_t* n_tokens,
                    const void* const* comp, const uint8_t* const* comp_scales,
                    const int32_t* idx, void* out, void* workspace, int32_t* dev_status,
                    void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* ws_o = static_cast<float*>(workspace);
    float2* ws_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + ws_o_bytes(B));
    const float scale_log2 = p->softmax_scale * kLog2e;
    const dim3 grid(kSplits, B);
    // loads the kernels and sets their shared-memory limits on this device, once per device
    if (const int rc = ensure_loaded()) return rc;
    if (quant) {
        k_sparse_attn_bf16<<<grid, kThreads, kSmemBf16, s>>>(
            static_cast<const __nv_bfloat16*>(q), win, n_tokens, comp, comp_scales, idx,
            p->compress_ratio, scale_log2, ws_o, ws_ml, dev_status, p->win_layout == CSA2_WIN_LINEAR);
        k_sparse_attn_merge<true><<<dim3(kH, B), 128, 0, s>>>(sink, ws_o, ws_ml, out);
    } else {
        k_sparse_attn_f32<<<grid, kF32Threads, kSmemF32, s>>>(
            static_cast<const float*>(q), win, n_tokens, comp, idx, p->compress_ratio, scale_log2,
            ws_o, ws_ml, dev_status, p->win_layout == CSA2_WIN_LINEAR);
        k_sparse_attn_merge<false><<<dim3(kH, B), 128, 0, s>>>(sink, ws_o, ws_ml, out);
    }
    return check_launch(name);
}
}  // namespace

extern "C" int csa2_sparse_attn(const csa2_params* p, int B, const void* q, const float* sink,
                                const void* const* win, const int32_t* n_tokens,
                                const void* const* comp, const uint8_t* const* comp_scales,
                                const int32_t* idx, void* out, void* workspace, size_t ws_bytes,
                                int32_t* dev_status, void* stream) {
    bool quant = false;
    const int rc = check_single("sparse_attn", p, B, q, sink, win, n_tokens, comp, comp_scales, idx,
                                out, workspace, ws_bytes, &quant);
    if (rc != CSA2_OK) return rc < 0 ? CSA2_OK : rc;
    if (quant)  // tcgen05, the fused kernel of sparse_attn_tc.cu with one layer
        return sparse_attn_tc_single("sparse_attn", p, B, q, sink, win, n_tokens, comp, comp_scales,
                                     idx, out, workspace, ws_bytes, dev_status, stream);
    return launch_split_kv("sparse_attn", p, B, false, q, sink, win, n_tokens, comp, comp_scales,
                           idx, out, workspace, dev_status, stream);
}

extern "C" int csa2_sparse_attn_mma(const csa2_params* p, int B, const void* q, const float* sink,
                                    const void* const* win, const int32_t* n_tokens,
                                    const void* const* comp, const uint8_t* const* comp_scales,
                                    const int32_t* idx, void* out, void* workspace, size_t ws_bytes,
                                    int32_t* dev_status, void* stream) {
    bool quant = false;
    const int rc = check_single("sparse_attn_mma", p, B, q, sink, win, n_tokens, comp, comp_scales,
                                idx, out, workspace, ws_bytes, &quant);
    if (rc != CSA2_OK) return rc < 0 ? CSA2_OK : rc;
    return launch_split_kv("sparse_attn_mma", p, B, quant, q, sink, win, n_tokens, comp,
                           comp_scales, idx, out, workspace, dev_status, stream);
}

// ---------------------------------------------------------------------------
// No-allocation variant. Its scratch (the partial results of csa2_sparse_attn's
// schedules) lives in this file-scope device array, so the caller passes no
// workspace. Some callers cannot allocate device memory at all: a serving engine
// that has already handed the free HBM to its own pool (the KV cache is sized to
// fill it), or a latency-critical path where a cudaMalloc/cudaFree would
// synchronise the device. The array holds the partials of at most
// kNoAllocMaxBatch sequences (the pages' serving batch, max-num-seqs 32): the
// fp32 split-KV passes need 32 x 657,920 B = 21,053,440 B, the tcgen05
// schedule of the quantised formats at most 31 cut units x 263,168 B + counts,
// and every GPU that loads the library holds the array until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {
constexpr int kNoAllocMaxBatch = 32;
constexpr size_t kNoAllocScratchBytes =
    (size_t)kNoAllocMaxBatch * csa2::kSplits * csa2::kH * (csa2::kD * sizeof(float) + sizeof(float2));
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

// the tcgen05 schedule's need for B <= 32: at most 31 boundary slots of two
// partials (64 x 512 outputs + 64 maxima + 64 sums, fp32) after 256 B of counts
static_assert(256 + 31 * 2 * (csa2::kH * csa2::kD + 2 * csa2::kH) * sizeof(float) <=
                  kNoAllocScratchBytes,
              "no-allocation scratch too small for the tcgen05 schedule");

static __device__ __align__(256) unsigned char g_sparse_attn_scratch[kNoAllocScratchBytes];

extern "C" int csa2_sparse_attn_noalloc(const csa2_params* p, int B, const void* q,
                                        const float* sink, const void* const* win,
                                        const int32_t* n_tokens, const void* const* comp,
                                        const uint8_t* const* comp_scales, const int32_t* idx,
                                        void* out, int32_t* dev_status, void* stream) {
    CSA2_CHECK_PARAMS(p);
    if (B < 0) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn_noalloc: negative batch");
    if (B > kNoAllocMaxBatch)
        return fail(CSA2_ERR_UNSUPPORTED,
                    "sparse_attn_noalloc: at most 32 sequences per call (the built-in scratch "
                    "holds 32); split the batch or use csa2_sparse_attn with a workspace");
    if (const int rc = ensure_loaded()) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return check_launch("sparse_attn_noalloc: current device");
    void* scratch = nullptr;
    {
        // once per device, with that device current: the device address of the array
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void* ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&ptr, g_sparse_attn_scratch);
            if (e != cudaSuccess || !ptr)
                return fail(CSA2_ERR_CUDA, std::string("sparse_attn_noalloc: scratch address: ") +
                                               cudaGetErrorString(e));
            g_noalloc_ptr[dev] = ptr;
        }
        scratch = g_noalloc_ptr[dev];
    }
    return csa2_sparse_attn(p, B, q, sink, win, n_tokens, comp, comp_scales, idx, out, scratch,
                            kNoAllocScratchBytes, dev_status, stream);
}
