// Two-level candidate selection.
// "DeepSeek-V4.1-Flash-NVFP4" §3.3 (select_candidate_blocks): compressed
// positions in blocks of 8, a block scored by its best position, the top-2048
// blocks kept with the block of the newest position always kept; then the
// top-512 positions inside the kept blocks.
//
// One CTA of 1024 threads per sequence. Each level is an exact radix select
// on order-preserving u32 keys (four 8-bit digit passes with a shared-memory
// histogram, the digit found by one warp's scan), then an ordered pass that
// takes the tied elements with the lowest indices. Level 2 works on a copy of
// the candidate keys in shared memory; its candidate list is ascending by
// position, so the output comes out ascending by construction.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCand = kKb * kBlk;  // 16384

struct SelShared {
    uint32_t hist[256];
    uint32_t warp_sum[kWarps];
    int32_t bcast[4];
    int32_t kept[kKb];
    uint32_t cand[kMaxCand];
};

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Exclusive prefix sum of one value per thread over the CTA (in thread order).
__device__ uint32_t block_excl_scan(uint32_t v, SelShared& sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t incl = warp_incl_scan(v);
    if (lane == 31) sh.warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t x = sh.warp_sum[lane];
        const uint32_t xi = warp_incl_scan(x);
        sh.warp_sum[lane] = xi - x;
    }
    __syncthreads();
    const uint32_t r = sh.warp_sum[warp] + incl - v;
    __syncthreads();
    return r;
}

// K-th largest key among n keys (1 <= K <= n). On return *need_eq is how many
// elements equal to the K-th key belong to the top K.
template <class KeyAt>
__device__ uint32_t radix_kth(int n, int K, KeyAt key_at, SelShared& sh, int* need_eq) {
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t prefix = 0, mask = 0;
    int remaining = K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (tid < 256) sh.hist[tid] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
            const uint32_t k = key_at(i);
            if ((k & mask) == prefix) atomicAdd(&sh.hist[(k >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns digits 255-8l down to 248-8l (largest digits first)
            uint32_t c[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = sh.hist[255 - 8 * lane - j];
                tot += c[j];
            }
            const uint32_t incl = warp_incl_scan(tot), excl = incl - tot;
            if (excl < (uint32_t)remaining && (uint32_t)remaining <= incl) {
                uint32_t acc = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (acc + c[j] >= (uint32_t)remaining) {
                        sh.bcast[0] = 255 - 8 * lane - j;
                        sh.bcast[1] = (int)acc;
                        break;
                    }
                    acc += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= (uint32_t)sh.bcast[0] << shift;
        mask |= 255u << shift;
        remaining -= sh.bcast[1];
        __syncthreads();
    }
    *need_eq = remaining;
    return prefix;
}

// Marks the top K of n keys (ties -> lower index) and writes the marked
// indices, in ascending order, through emit(rank, i). Each thread owns a
// contiguous chunk of indices so that tie ranks follow index order.
template <class KeyAt, class Emit>
__device__ void select_top(int n, int K, KeyAt key_at, Emit emit, SelShared& sh) {
    int need_eq;
    const uint32_t kth = radix_kth(n, K, key_at, sh, &need_eq);
    const int chunk = (n + kThreads - 1) / kThreads;
    const int i0 = min(n, (int)threadIdx.x * chunk), i1 = min(n, i0 + chunk);
    uint32_t n_eq = 0;
    for (int i = i0; i < i1; ++i) n_eq += key_at(i) == kth;
    uint32_t eq_rank = block_excl_scan(n_eq, sh);
    uint32_t n_sel = 0;
    {
        uint32_t r = eq_rank;
        for (int i = i0; i < i1; ++i) {
            const uint32_t k = key_at(i);
            n_sel += (k > kth) || (k == kth && r++ < (uint32_t)need_eq);
        }
    }
    uint32_t out = block_excl_scan(n_sel, sh);
    for (int i = i0; i < i1; ++i) {
        const uint32_t k = key_at(i);
        if ((k > kth) || (k == kth && eq_rank++ < (uint32_t)need_eq)) emit(out++, i);
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
k_select_topk(int64_t max_ncomp, int ratio, const float* __restrict__ scores,
              const float* __restrict__ block_max, const int32_t* __restrict__ n_tokens,
              int32_t* idx, int32_t* n_sel_out, int32_t* dev_status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
    const int b = blockIdx.x, tid = threadIdx.x;
    int64_t n_c64 = n_tokens[b] / ratio;
    if (n_c64 > max_ncomp || n_c64 < 0) {
        if (tid == 0) raise_status(dev_status, CSA2_DEV_BAD_LENGTH);
        n_c64 = n_c64 < 0 ? 0 : max_ncomp;
    }
    const int n_c = (int)n_c64;
    const int64_t ld_b = (max_ncomp + kBlk - 1) / kBlk;
    const float* bm = block_max + (int64_t)b * ld_b;
    const float* sc = scores + (int64_t)b * max_ncomp;
    int32_t* out = idx + (int64_t)b * kKp;
    const int n_b = (n_c + kBlk - 1) / kBlk;

    // ---- level 1: kept blocks, ascending ----
    int n_kept;
    if (n_b <= kKb) {
        for (int i = tid; i < n_b; i += kThreads) sh.kept[i] = i;
        n_kept = n_b;
    } else {
        // best K_b - 1 among blocks [0, n_b - 1), then the newest block n_b - 1
        select_top(
            n_b - 1, kKb - 1, [&](int i) { return score_key(bm[i]); },
            [&](uint32_t r, int i) { sh.kept[r] = i; }, sh);
        if (tid == 0) sh.kept[kKb - 1] = n_b - 1;
        n_kept = kKb;
    }
    __syncthreads();

    // ---- level 2: positions of the kept blocks ----
    // the last kept block is block n_b - 1, the only one that may be partial
    const int n_cand = n_kept == 0 ? 0 : (n_kept - 1) * kBlk + (n_c - (n_b - 1) * kBlk);
    for (int i = tid; i < n_cand; i += kThreads)
        sh.cand[i] = score_key(sc[sh.kept[i / kBlk] * kBlk + (i % kBlk)]);
    for (int i = tid; i < kKp; i += kThreads) out[i] = -1;
    __syncthreads();
    if (n_cand <= kKp) {
        for (int i = tid; i < n_cand; i += kThreads) out[i] = sh.kept[i / kBlk] * kBlk + i % kBlk;
    } else {
        select_top(
            n_cand, kKp, [&](int i) { return sh.cand[i]; },
            [&](uint32_t r, int i) { out[r] = sh.kept[i / kBlk] * kBlk + i % kBlk; }, sh);
    }
    if (tid == 0 && n_sel_out) n_sel_out[b] = min(n_cand, kKp);
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" int csa2_select_topk(const csa2_params* p, int B, int64_t max_ncomp,
                                const float* scores, const float* block_max,
                                const int32_t* n_tokens, int32_t* idx, int32_t* n_sel,
                                int32_t* dev_status, void* stream) {
    CSA2_CHECK_PARAMS(p);
    if (B < 0 || max_ncomp < 0) return fail(CSA2_ERR_INVALID_ARG, "select_topk: negative size");
    if (B == 0) return CSA2_OK;
    if (p->block_size != kBlk || p->topk_blocks != kKb || p->topk_pos != kKp ||
        p->compress_ratio < 1)
        return fail(CSA2_ERR_UNSUPPORTED, "select_topk: built for blocks of 8, 2048 blocks, 512");
    if (max_ncomp > 0x7fffffffLL)
        return fail(CSA2_ERR_UNSUPPORTED, "select_topk: more than 2^31 positions");
    if (!scores || !block_max || !n_tokens || !idx)
        return fail(CSA2_ERR_INVALID_ARG, "select_topk: NULL buffer");
    static bool attr_set = false;
    const int smem = (int)sizeof(SelShared);
    if (!attr_set) {
        if (cudaFuncSetAttribute(k_select_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem) != cudaSuccess)
            return check_launch("select_topk: smem attribute");
        attr_set = true;
    }
    k_select_topk<<<B, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
        max_ncomp, p->compress_ratio, scores, block_max, n_tokens, idx, n_sel, dev_status);
    return check_launch("select_topk");
}
