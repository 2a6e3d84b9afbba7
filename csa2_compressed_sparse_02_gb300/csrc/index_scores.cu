// Decode Indexer with fused block maximum.
// "DeepSeek-V4.1-Flash-NVFP4" §3.3: 32 FP4 index query heads score the shared
// FP4 index key; ReLU, per-head weights, sum; blocks of 8 positions are scored
// by their best position.
//
// CUDA-core build: one thread per key, 32 fp32 accumulators (one per head),
// the query decoded once per CTA into shared memory as [dim][head] so that a
// warp reads it by broadcast. Exact for the inputs the header describes
// (every partial sum representable), so the fp32 result does not depend on
// the order of the adds.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kKeysPerCta = 256;

__global__ void __launch_bounds__(kKeysPerCta)
k_index_scores_cc(int64_t max_ncomp, int ratio, const uint8_t* __restrict__ q_vals,
                  const uint8_t* __restrict__ q_scales, const float* __restrict__ w,
                  const uint8_t* const* key_vals, const uint8_t* const* key_scales,
                  const int32_t* __restrict__ n_tokens, float* scores, float* block_max,
                  int32_t* dev_status) {
    __shared__ float4 sq[kDi][kHi / 4];  // sq[d][h/4] = q[h..h+3][d]
    __shared__ float sw[kHi];
    const int b = blockIdx.y, tid = threadIdx.x;
    int64_t n_c = n_tokens[b] / ratio;
    if (n_c > max_ncomp || n_c < 0) {
        if (tid == 0 && blockIdx.x == 0) raise_status(dev_status, CSA2_DEV_BAD_LENGTH);
        n_c = n_c < 0 ? 0 : max_ncomp;
    }
    const int64_t t0 = (int64_t)blockIdx.x * kKeysPerCta;
    if (t0 >= n_c) return;

    float* sqf = reinterpret_cast<float*>(sq);
    const uint8_t* qv = q_vals + (int64_t)b * kHi * (kDi / 2);
    const uint8_t* qs = q_scales + (int64_t)b * kHi * (kDi / kGroup);
    for (int e = tid; e < kHi * kDi / 2; e += kKeysPerCta) {  // one byte = 2 dims
        const int h = e / (kDi / 2), d = 2 * (e % (kDi / 2));
        const float s = e4m3_value(qs[h * (kDi / kGroup) + d / kGroup]);
        const uint32_t h2 = e2m1x2_to_half2(qv[e]);
        sqf[d * kHi + h] = __half2float(__ushort_as_half((uint16_t)(h2 & 0xffff))) * s;
        sqf[(d + 1) * kHi + h] = __half2float(__ushort_as_half((uint16_t)(h2 >> 16))) * s;
    }
    if (tid < kHi) sw[tid] = w[(int64_t)b * kHi + tid];
    __syncthreads();

    const int64_t t = t0 + tid;
    const bool valid = t < n_c;
    float acc[kHi];
#pragma unroll
    for (int h = 0; h < kHi; ++h) acc[h] = 0.0f;
    if (valid) {
        const uint4* kp = reinterpret_cast<const uint4*>(key_vals[b] + t * (kDi / 2));
        const uint2 ks = *reinterpret_cast<const uint2*>(key_scales[b] + t * (kDi / kGroup));
        const uint32_t sc[2] = {ks.x, ks.y};
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {  // 16 bytes = 32 dims = 2 groups
            const uint4 kb = kp[q4];
            const uint32_t words[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const int g = 2 * q4 + wi / 2;
                const float s = e4m3_value((uint8_t)(sc[g / 4] >> (8 * (g % 4))));
#pragma unroll
                for (int bi = 0; bi < 4; ++bi) {
                    const int d = 32 * q4 + 8 * wi + 2 * bi;
                    const uint32_t h2 = e2m1x2_to_half2((words[wi] >> (8 * bi)) & 0xffu);
                    const float k0 = __half2float(__ushort_as_half((uint16_t)(h2 & 0xffff))) * s;
                    const float k1 = __half2float(__ushort_as_half((uint16_t)(h2 >> 16))) * s;
#pragma unroll
                    for (int hq = 0; hq < kHi / 4; ++hq) {
                        const float4 a = sq[d][hq];
                        acc[4 * hq + 0] = __fmaf_rn(a.x, k0, acc[4 * hq + 0]);
                        acc[4 * hq + 1] = __fmaf_rn(a.y, k0, acc[4 * hq + 1]);
                        acc[4 * hq + 2] = __fmaf_rn(a.z, k0, acc[4 * hq + 2]);
                        acc[4 * hq + 3] = __fmaf_rn(a.w, k0, acc[4 * hq + 3]);
                    }
#pragma unroll
                    for (int hq = 0; hq < kHi / 4; ++hq) {
                        const float4 a = sq[d + 1][hq];
                        acc[4 * hq + 0] = __fmaf_rn(a.x, k1, acc[4 * hq + 0]);
                        acc[4 * hq + 1] = __fmaf_rn(a.y, k1, acc[4 * hq + 1]);
                        acc[4 * hq + 2] = __fmaf_rn(a.z, k1, acc[4 * hq + 2]);
                        acc[4 * hq + 3] = __fmaf_rn(a.w, k1, acc[4 * hq + 3]);
                    }
                }
            }
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int h = 0; h < kHi; ++h) s = __fmaf_rn(sw[h], acc[h] > 0.0f ? acc[h] : 0.0f, s);
    if (valid) scores[(int64_t)b * max_ncomp + t] = s;
    float m = valid ? s : -INFINITY;
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    if (valid && (tid & (kBlk - 1)) == 0)
        block_max[(int64_t)b * ((max_ncomp + kBlk - 1) / kBlk) + t / kBlk] = m;
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" int csa2_index_scores(const csa2_params* p, int B, int64_t max_ncomp,
                                 const uint8_t* q_vals, const uint8_t* q_scales, const float* w,
                                 const uint8_t* const* key_vals, const uint8_t* const* key_scales,
                                 const int32_t* n_tokens, float* scores, float* block_max,
                                 int32_t* dev_status, void* stream) {
    CSA2_CHECK_PARAMS(p);
    if (B < 0 || max_ncomp < 0) return fail(CSA2_ERR_INVALID_ARG, "index_scores: negative size");
    if (B == 0 || max_ncomp == 0) return CSA2_OK;
    if (p->index_heads != kHi || p->index_dim != kDi || p->block_size != kBlk ||
        p->compress_ratio < 1)
        return fail(CSA2_ERR_UNSUPPORTED, "index_scores: built for 32 heads x 128, blocks of 8");
    if (!q_vals || !q_scales || !w || !key_vals || !key_scales || !n_tokens || !scores ||
        !block_max)
        return fail(CSA2_ERR_INVALID_ARG, "index_scores: NULL buffer");
    const int64_t gx = (max_ncomp + kKeysPerCta - 1) / kKeysPerCta;
    if (gx > 0x7fffffff) return fail(CSA2_ERR_UNSUPPORTED, "index_scores: too many positions");
    k_index_scores_cc<<<dim3((unsigned)gx, B), kKeysPerCta, 0, static_cast<cudaStream_t>(stream)>>>(
        max_ncomp, p->compress_ratio, q_vals, q_scales, w, key_vals, key_scales, n_tokens, scores,
        block_max, dev_status);
    return check_launch("index_scores");
}
