// Two-level candidate selection.
// "DeepSeek-V4.1-Flash-NVFP4" §3.3 (select_candidate_blocks): compressed
// positions in blocks of 8, a block scored by its best position, the top-2048
// blocks kept with the block of the newest position always kept; then the
// top-512 positions inside the kept blocks.
//
// With the block score the best position's score and 2,047 > 512, that rule
// returns the 512 best positions of the sequence, and they lie in the 512 best
// blocks (see k_select_topk). So level 1 here keeps the 512 best blocks and
// level 2 selects among their at most 4,096 positions: the same positions,
// found with a quarter of the block keys kept and of the scores gathered.
//
// One CTA of 1024 threads per sequence, or, for a small batch, a cluster of 4
// CTAs per sequence whose level-1 pass over the block maxima is split in
// quarters (counts and candidates exchanged through distributed shared memory,
// every wait bounded), CTA 0 finishing alone. Each level is an exact radix select
// on order-preserving u32 keys (four 8-bit digit passes with a shared-memory
// histogram, the digit found by one warp's scan), then an ordered pass that
// takes the tied elements with the lowest indices. Level 2 works on a copy of
// the candidate keys in shared memory; its candidate list is ascending by
// position, so the output comes out ascending by construction.
//
// Level 1 keeps 512 of up to 131,072 blocks, so it first narrows the field:
// a threshold estimated from a strided sample of 2,048 block maxima and one pass
// that keeps the blocks at or above it (in index order, in shared memory). The
// top 512 blocks all lie at or above any threshold that at least 512 blocks
// reach, and so do the 512 best positions (each scores at least the 512th best
// block maximum). So the common path goes flat from there: the positions of at
// most 2,048 candidate blocks are gathered into shared memory, those at or above
// the threshold kept (usually a few hundred more than 512), and one exact select
// of 512 runs among them. When the count falls outside [512, kMaxFiltered] the
// threshold moves, and after a few tries the exact select runs over all blocks
// in global memory; with more than 2,048 candidate blocks, or more than 4,096
// tied positions at or above the threshold, the 512 best candidate blocks are
// selected first and level 2 keeps the positions at or above the 512th block's
// maximum before its exact select.
#include "common.cuh"
#include "sm100.cuh"

namespace csa2 {
namespace {
using namespace sm100;

constexpr int kSample = 2048;
constexpr int kMaxFiltered2 = kKp * kBlk;  // level 2: every candidate of the kKp kept blocks
constexpr int kStagePerWarp = 256;   // kept pairs a warp stages during the vector filter's pass
constexpr int kClMax = 4;            // CTAs of one sequence in the cluster launch
constexpr int kAttempts = 4;         // thresholds tried before the exact select over every block

// Two builds: 1,024 threads and up to 8,192 level-1 candidates (159 KB of shared
// memory: one CTA per SM) for the cluster launch and batches that fill one wave;
// 512 threads and up to 4,096 candidates (91 KB: two CTAs per SM, so that one CTA's
// barriers and memory round trips overlap the other's work) for larger batches.
template <int NT, int MF>
struct SelCfg {
    static constexpr int kThreads = NT;
    static constexpr int kWarps = NT / 32;
    static constexpr int kMaxFiltered = MF;
    static constexpr int kMaxCand = MF + kSample;  // level 1: filtered keys, sample at the end
    static constexpr int kStage = kWarps * kStagePerWarp;  // pairs the level-1 filter can stage
    static constexpr int kFlatCap = 2 * kStage;  // positions the flat pass gathers (the whole stage area)
};
using SelWide = SelCfg<1024, 8192>;
using SelHalf = SelCfg<512, 4096>;

// the configuration's sizes under their short names, in every function below
#define SEL_CFG_NAMES                                      \
    constexpr int kThreads = C::kThreads;                  \
    constexpr int kWarps = C::kWarps;                      \
    constexpr int kMaxFiltered = C::kMaxFiltered;          \
    constexpr int kMaxCand = C::kMaxCand;                  \
    constexpr int kStage = C::kStage;                      \
    constexpr int kFlatCap = C::kFlatCap;                  \
    (void)kThreads, (void)kWarps, (void)kMaxFiltered, (void)kMaxCand, (void)kStage, (void)kFlatCap

template <class C>
struct SelShared {
    uint32_t hist[256];
    uint32_t warp_sum[C::kWarps];
    int32_t bcast[4];
    int32_t kept[kKp];
    uint32_t cand[C::kMaxCand];        // level 1: filtered keys (sample at the end); level 2 keys
    int32_t cand_idx[C::kMaxFiltered];  // index of each filtered key
    uint32_t cand2[kMaxFiltered2];   // level 2 filtered keys
    // level 1 filter: kept (key, index) pairs per warp, in order (keys in
    // [0, kStage), indices in [kStage, 2 kStage)); the flat pass: position keys
    uint32_t stage[2 * C::kStage];
    // cluster launch: each CTA's level-1 candidate count, per attempt, written into
    // every CTA of the cluster; cnt_bar completes a phase per attempt once all CTAs
    // wrote theirs, gat_bar (CTA 0) once the others copied their candidates in
    uint32_t cl_cnt[kAttempts][kClMax];
    uint64_t cnt_bar, gat_bar;
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

// K-th largest key among n keys (1 <= K <= n). On return *need_eq is how many
// elements equal to the K-th key belong to the top K.
// With digits < 4 only the top 8*digits bits are resolved: the result is the
// K-th largest key with its low bits cleared, a lower bound that at least K keys
// reach (used as a filter threshold).
template <class C, class KeyAt>
__device__ uint32_t radix_kth(int n, int K, KeyAt key_at, SelShared<C>& sh, int* need_eq,
                              int digits = 4) {
    SEL_CFG_NAMES;
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t prefix = 0, mask = 0;
    int remaining = K;
    for (int shift = 24; shift >= 32 - 8 * digits; shift -= 8) {
        if (tid < 256) sh.hist[tid] = 0;
        __syncthreads();
        // warp-aggregated: one shared atomic per distinct digit per warp (scores share
        // sign and exponent, so most keys of a pass land in very few bins)
        for (int base = 0; base < n; base += kThreads) {
            const int i = base + tid;
            const uint32_t k = i < n ? key_at(i) : 0u;
            const bool active = i < n && (k & mask) == prefix;
            const uint32_t am = __ballot_sync(0xffffffffu, active);
            if (active) {
                const uint32_t d = (k >> shift) & 255u;
                const uint32_t peers = __match_any_sync(am, d);
                if (lane == __ffs(peers) - 1) atomicAdd(&sh.hist[d], (uint32_t)__popc(peers));
            }
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

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan of one value per warp (lane 0 holds it) over the CTA's warps;
// every lane of warp w receives the sum over warps < w. *total gets the sum.
template <class C>
__device__ uint32_t warp_excl_scan(uint32_t v, SelShared<C>& sh, uint32_t* total) {
    SEL_CFG_NAMES;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sh.warp_sum[warp] = v;
    __syncthreads();
    if (warp == 0) {  // lanes past the CTA's warp count add nothing
        const uint32_t x = lane < kWarps ? sh.warp_sum[lane] : 0u;
        const uint32_t xi = warp_incl_scan(x);
        if (lane < kWarps) sh.warp_sum[lane] = xi - x;
        if (lane == 31) sh.bcast[3] = (int)xi;
    }
    __syncthreads();
    const uint32_t r = sh.warp_sum[warp];
    *total = (uint32_t)sh.bcast[3];
    __syncthreads();
    return r;
}

// Marks the top K of n keys (ties -> lower index) and writes the marked
// indices, in ascending order, through emit(rank, i). Each warp owns a
// contiguous range of indices and walks it 32 at a time (coalesced), so tie
// ranks and output ranks follow index order via ballots.
template <class C, class KeyAt, class Emit>
__device__ uint32_t select_top(int n, int K, KeyAt key_at, Emit emit, SelShared<C>& sh) {
    SEL_CFG_NAMES;
    int need_eq;
    const uint32_t kth = radix_kth(n, K, key_at, sh, &need_eq);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = lanemask_lt();
    const int R = (n + kWarps - 1) / kWarps;
    const int w0 = min(n, warp * R), w1 = min(n, w0 + R);
    uint32_t n_gt = 0, n_eq = 0;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < w1 ? key_at(i) : 0u;
        n_gt += __popc(__ballot_sync(0xffffffffu, i < w1 && k > kth));
        n_eq += __popc(__ballot_sync(0xffffffffu, i < w1 && k == kth));
    }
    uint32_t tot;
    const uint32_t eq_off = warp_excl_scan(n_eq, sh, &tot);
    const int take_eq = max(0, min((int)n_eq, need_eq - (int)eq_off));
    uint32_t out = warp_excl_scan(n_gt + (uint32_t)take_eq, sh, &tot);
    uint32_t r_eq = eq_off;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < w1 ? key_at(i) : 0u;
        const bool gt = i < w1 && k > kth, eq = i < w1 && k == kth;
        const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
        const bool take = gt || (eq && r_eq + __popc(eqm & lt) < (uint32_t)need_eq);
        const uint32_t tm = __ballot_sync(0xffffffffu, take);
        if (take) emit(out + __popc(tm & lt), i);
        out += __popc(tm);
        r_eq += __popc(eqm);
    }
    __syncthreads();
    return kth;
}


// Keys at or above thr among key_at(0..n), kept in index order: (key, index)
// pairs written to keys_out/idx_out (capacity cap). Each warp walks its own
// contiguous range, 8 x 32 elements per round with the loads issued first.
// Returns the count (which may exceed cap: then nothing was written).
template <class C, class KeyAt>
__device__ int filter_ge(int n, uint32_t thr, KeyAt key_at, uint32_t* keys_out, int32_t* idx_out,
                         int cap, SelShared<C>& sh) {
    SEL_CFG_NAMES;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = lanemask_lt();
    const int R = (n + kWarps - 1) / kWarps;
    const int w0 = min(n, warp * R), w1 = min(n, w0 + R);
    constexpr int U = 8;
    uint32_t c = 0;
    for (int base = w0; base < w1; base += 32 * U) {
        uint32_t k[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + 32 * u + lane;
            k[u] = i < w1 ? key_at(i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + 32 * u + lane;
            c += __popc(__ballot_sync(0xffffffffu, i < w1 && k[u] >= thr));
        }
    }
    uint32_t total;
    uint32_t o = warp_excl_scan(c, sh, &total);
    if ((int)total > cap) return (int)total;
    for (int base = w0; base < w1; base += 32 * U) {
        uint32_t k[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + 32 * u + lane;
            k[u] = i < w1 ? key_at(i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + 32 * u + lane;
            const bool keep = i < w1 && k[u] >= thr;
            const uint32_t m = __ballot_sync(0xffffffffu, keep);
            if (keep) {
                keys_out[o + __popc(m & lt)] = k[u];
                idx_out[o + __popc(m & lt)] = i;
            }
            o += __popc(m);
        }
    }
    __syncthreads();
    return (int)total;
}

// filter_ge over n block maxima read straight from global memory, for a
// 16-byte aligned row. One pass of 16-byte loads (8 in flight per thread):
// every warp walks its own contiguous range of 128-element chunks (lane l
// covers elements 4l..4l+3 of a chunk) and stages its kept (key, index) pairs,
// in index order, in its own slot of kStagePerWarp; a prefix over the warps'
// counts then places every slot. Returns -1 when a slot overflowed (the caller
// then uses filter_ge), else the count (which may exceed cap: then nothing was
// written).
template <class C>
__device__ int filter_ge_vec(int n, uint32_t thr, const float* __restrict__ bm, uint32_t* keys_out,
                             int32_t* idx_out, int cap, SelShared<C>& sh) {
    SEL_CFG_NAMES;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunks = (n + 127) / 128;
    const int R = (chunks + kWarps - 1) / kWarps;
    const int c0 = min(chunks, warp * R), c1 = min(chunks, c0 + R);
    uint32_t* skey = sh.stage + warp * kStagePerWarp;
    int32_t* sidx = reinterpret_cast<int32_t*>(sh.stage + kStage) + warp * kStagePerWarp;
    // the value whose key is thr: key >= thr <=> value >= thr_f (keys are monotone)
    const uint32_t tb = (thr & 0x80000000u) ? (thr & 0x7fffffffu) : ~thr;
    const float thr_f = __uint_as_float(tb);
    constexpr int U = 8;
    uint32_t cnt = 0;
    // one chunk's four values of this lane -> kept flags, staged pairs, count
    auto chunk = [&](int cbu, float4 v) {
        const int e = 128 * cbu + 4 * lane;
        const int left = n - e;  // elements of this lane's four inside n
        const uint32_t valid = left >= 4 ? 15u : (left > 0 ? (1u << left) - 1u : 0u);
        const uint32_t m4 = valid & ((uint32_t)(v.x >= thr_f) | ((uint32_t)(v.y >= thr_f) << 1) |
                                     ((uint32_t)(v.z >= thr_f) << 2) | ((uint32_t)(v.w >= thr_f) << 3));
        const uint32_t c = __popc(m4);
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        uint32_t at = cnt + incl - c;
        if (m4) {
            const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if ((m4 >> q) & 1u) {
                    if (at < (uint32_t)kStagePerWarp) {
                        skey[at] = score_key(f[q]);
                        sidx[at] = e + q;
                    }
                    ++at;
                }
            }
        }
        cnt += __shfl_sync(0xffffffffu, incl, 31);
    };
    // whole batches of U chunks inside n: the loads carry no condition
    const int c_full = min(c1, n / 128);  // chunks entirely inside n
    int cb = c0;
    for (; cb + U <= c_full; cb += U) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = __ldg(reinterpret_cast<const float4*>(bm + 128 * (cb + u) + 4 * lane));
#pragma unroll
        for (int u = 0; u < U; ++u) chunk(cb + u, v[u]);
    }
    for (; cb < c1; ++cb) {  // the rest, one chunk at a time, loads guarded
        const int e = 128 * cb + 4 * lane;
        float4 v;
        if (e + 3 < n) {
            v = __ldg(reinterpret_cast<const float4*>(bm + e));
        } else {
            v.x = e < n ? bm[e] : -INFINITY;
            v.y = e + 1 < n ? bm[e + 1] : -INFINITY;
            v.z = e + 2 < n ? bm[e + 2] : -INFINITY;
            v.w = -INFINITY;
        }
        chunk(cb, v);
    }
    uint32_t total;
    const uint32_t o = warp_excl_scan(cnt, sh, &total);  // (its barriers also publish the stages)
    sh.bcast[2] = 0;
    __syncthreads();
    if (cnt > (uint32_t)kStagePerWarp && lane == 0) sh.bcast[2] = 1;
    __syncthreads();
    if (sh.bcast[2]) return -1;
    if ((int)total > cap) return (int)total;
    for (uint32_t i = lane; i < cnt; i += 32) {
        keys_out[o + i] = skey[i];
        idx_out[o + i] = sidx[i];
    }
    __syncthreads();
    return (int)total;
}

// ncl CTAs per sequence (1, or kClMax in a cluster launch): with a cluster, every
// CTA filters a quarter of the block maxima at level 1 and CTA 0 (rank 0 of the
// cluster) finishes the sequence alone once the others have copied their
// candidates into its shared memory.
template <class C>
__global__ void __launch_bounds__(C::kThreads, 1024 / C::kThreads)
k_select_topk(int64_t max_ncomp, int ratio, const float* __restrict__ scores,
              const float* __restrict__ block_max, const int32_t* __restrict__ n_tokens,
              int32_t* idx, int32_t* n_sel_out, int32_t* dev_status, int ncl) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SEL_CFG_NAMES;
    SelShared<C>& sh = *reinterpret_cast<SelShared<C>*>(smem_raw);
    const int b = blockIdx.x / ncl, tid = threadIdx.x;
    const int rank = ncl > 1 ? (int)cluster_ctarank() : 0;
    trace_start(kTraceSelect);
    // the attention after it may be scheduled now (it waits for this grid first)
    grid_dep_launch_dependents();
    if (ncl > 1) {
        if (tid == 0) {
            mbar_init(&sh.cnt_bar, (uint32_t)ncl);
            mbar_init(&sh.gat_bar, (uint32_t)(ncl - 1));
            fence_mbar_init();
        }
        // every CTA of the cluster has started and initialised its barriers before
        // any of them touches another's shared memory
        cluster_sync_all();
    }
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

    // The two levels' result is the kKp best positions of the sequence by (score
    // desc, position asc): a best position's block ranks at least as high as the
    // position itself (its block maximum is at least its score, ties going to the
    // lower block as to the lower position), so the blocks holding the kKp best
    // positions are the top of the block order, and the kKb - 1 best blocks other
    // than the newest (kKb - 1 >= kKp) hold all of them whatever the newest block
    // scores. The kernel therefore keeps the kKp best blocks (over all blocks) and
    // selects among their at most 8 kKp positions, which gives the same positions
    // as keeping kKb blocks and selecting among 8 kKb.
    // ---- level 1: the kKp best blocks, ascending ----
    int n_kept;
    uint32_t thr2 = 0u;  // a key the kKp-th best position reaches
    if (n_b <= kKp) {
        if (rank > 0) return;  // the cluster's other CTAs have nothing to do
        for (int i = tid; i < n_b; i += kThreads) sh.kept[i] = i;
        n_kept = n_b;
    } else {
        const int K1 = kKp;
        // this CTA's blocks [lo, hi): whole 128-block chunks, so bm + lo stays 16-byte aligned
        const int span = ((n_b + ncl - 1) / ncl + 127) / 128 * 128;
        const int lo = min(n_b, rank * span), hi = min(n_b, lo + span);
        const bool vec_ok = (reinterpret_cast<uintptr_t>(bm) & 15u) == 0;
        // (a) threshold from a strided sample of all n_b blocks: the r-th largest sample
        //     key, r chosen so that about 1.5 K1 blocks reach it (every CTA of a cluster
        //     computes the same one)
        for (int i = tid; i < kSample; i += kThreads)
            sh.cand[kMaxCand - kSample + i] = score_key(bm[(int64_t)i * n_b / kSample]);
        __syncthreads();
        int r = (int)(1.5f * K1 * kSample / n_b) + 1;
        bool done = false;
        for (int attempt = 0; attempt < kAttempts && !done; ++attempt) {
            r = max(1, min(kSample, r));
            int unused;
            // the top 16 bits of the r-th largest sample key: a slightly lower threshold
            const uint32_t thr = radix_kth(kSample, r, [&](int i) { return sh.cand[kMaxCand - kSample + i]; },
                                           sh, &unused, 2);
            // (b) this CTA's blocks at or above it, in index order (indices from lo)
            const float* bml = bm + lo;
            int mine = vec_ok ? filter_ge_vec(hi - lo, thr, bml, sh.cand, sh.cand_idx, kMaxFiltered, sh) : -1;
            if (mine < 0)
                mine = filter_ge(
                    hi - lo, thr, [&](int i) { return score_key(bml[i]); }, sh.cand, sh.cand_idx,
                    kMaxFiltered, sh);
            // (c) the count over the cluster, the same in every CTA
            int total = mine, before = 0;
            if (ncl > 1) {
                if (tid == 0) {
                    const uint32_t slot = smem_u32(&sh.cl_cnt[attempt][rank]);
                    for (int m = 0; m < ncl; ++m) st_cluster_u32(mapa_shared(slot, (uint32_t)m), (uint32_t)mine);
                    for (int m = 0; m < ncl; ++m) mbar_arrive_cluster(mapa_shared(smem_u32(&sh.cnt_bar), (uint32_t)m));
                }
                if (!mbar_wait_cluster(&sh.cnt_bar, (uint32_t)(attempt & 1))) {
                    if (tid == 0) raise_status(dev_status, CSA2_DEV_TIMEOUT);
                    return;
                }
                total = 0;
                for (int m = 0; m < ncl; ++m) {
                    const int c = (int)sh.cl_cnt[attempt][m];
                    if (m < rank) before += c;
                    total += c;
                }
            }
            if (total < K1) {          // threshold too high: take a lower sample rank
                r = r * 2 + 8;
                continue;
            }
            if (total > kMaxFiltered) {  // too many candidates: take a higher sample rank
                if (r <= 1) break;
                r = r / 2;
                continue;
            }
            if (ncl > 1) {
                // (d) the candidates of CTA k go to CTA 0 at the count of CTAs < k (CTA 0's
                //     own are in place), in index order
                if (rank > 0) {
                    for (int i = tid; i < mine; i += kThreads) {
                        st_cluster_u32(mapa_shared(smem_u32(&sh.cand[before + i]), 0u), sh.cand[i]);
                        st_cluster_u32(mapa_shared(smem_u32(&sh.cand_idx[before + i]), 0u),
                                       (uint32_t)(sh.cand_idx[i] + lo));
                    }
                    asm volatile("fence.acq_rel.cluster;\n" ::: "memory");
                    __syncthreads();
                    if (tid == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sh.gat_bar), 0u));
                    return;
                }
                if (!mbar_wait_cluster(&sh.gat_bar, 0u)) {
                    if (tid == 0) raise_status(dev_status, CSA2_DEV_TIMEOUT);
                    return;
                }
            }
            // (e) flat: the candidate blocks hold every position of the kKp best (those
            //     score at least the kKp-th best block maximum, which is at least thr), so
            //     the kKp best of their positions at or above thr are the answer. Slot i =
            //     position i % 8 of candidate block i / 8, ascending by position; positions
            //     past n_c take the lowest key, and thr is above it.
            __syncthreads();
            auto vpos = [&](int i) { return sh.cand_idx[i >> 3] * kBlk + (i & (kBlk - 1)); };
            if (thr > 0u && total * kBlk <= kFlatCap) {
                const int nv = total * kBlk;
                if ((reinterpret_cast<uintptr_t>(sc) & 15u) == 0) {
                    // a block is 8 consecutive scores (32 bytes): two 16-byte loads
                    for (int q = tid; q < 2 * total; q += kThreads) {
                        const int i = 4 * q, pos = vpos(i);
                        if (pos + 3 < n_c) {
                            const float4 v = __ldg(reinterpret_cast<const float4*>(sc + pos));
                            *reinterpret_cast<uint4*>(&sh.stage[i]) =
                                make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
                        } else {
                            for (int c = 0; c < 4; ++c) sh.stage[i + c] = pos + c < n_c ? score_key(sc[pos + c]) : 0u;
                        }
                    }
                } else {
                    for (int i = tid; i < nv; i += kThreads) {
                        const int pos = vpos(i);
                        sh.stage[i] = pos < n_c ? score_key(sc[pos]) : 0u;
                    }
                }
                __syncthreads();
                // kept keys to cand2, their slots to the block keys' array (not needed on
                // this path; untouched when the filter overflows)
                int32_t* slot = reinterpret_cast<int32_t*>(sh.cand);
                const int n2 = filter_ge(
                    nv, thr, [&](int i) { return sh.stage[i]; }, sh.cand2, slot, kMaxFiltered2, sh);
                if (n2 <= kMaxFiltered2) {  // at least total >= kKp: each candidate block's maximum
                    select_top(
                        n2, kKp, [&](int i) { return sh.cand2[i]; },
                        [&](uint32_t rank_, int i) { out[rank_] = vpos(slot[i]); }, sh);
                    if (tid == 0 && n_sel_out) n_sel_out[b] = kKp;
                    trace_end(kTraceSelect);
                    return;
                }
            }
            // too many positions at or above thr (ties): the kKp best blocks first
            thr2 = select_top(
                total, K1, [&](int i) { return sh.cand[i]; },
                [&](uint32_t rank_, int i) { sh.kept[rank_] = sh.cand_idx[i]; }, sh);
            done = true;
        }
        if (!done) {  // exact select over every block, read from global memory (CTA 0)
            if (rank > 0) return;
            __syncthreads();
            thr2 = select_top(
                n_b, K1, [&](int i) { return score_key(bm[i]); },
                [&](uint32_t rank_, int i) { sh.kept[rank_] = i; }, sh);
        }
        n_kept = K1;
    }
    __syncthreads();

    // ---- level 2: positions of the kept blocks (block n_b - 1, the only one that
    // may be partial, comes last when kept) ----
    const int n_cand = n_kept == 0 ? 0
                                   : n_kept * kBlk - (sh.kept[n_kept - 1] == n_b - 1 ? n_b * kBlk - n_c : 0);
    if ((reinterpret_cast<uintptr_t>(sc) & 15u) == 0) {
        // blocks are 8 consecutive scores (32 bytes): two 16-byte loads per block
        for (int q = tid; q < 2 * n_kept; q += kThreads) {
            const int i = 4 * q;  // candidate index of the load's first score
            const int64_t pos = (int64_t)sh.kept[i / kBlk] * kBlk + (i % kBlk);
            if (i + 3 < n_cand) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(sc + pos));
                *reinterpret_cast<uint4*>(&sh.cand[i]) =
                    make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
            } else {
                for (int c = 0; c < 4 && i + c < n_cand; ++c) sh.cand[i + c] = score_key(sc[pos + c]);
            }
        }
    } else {
        for (int i = tid; i < n_cand; i += kThreads)
            sh.cand[i] = score_key(sc[sh.kept[i / kBlk] * kBlk + (i % kBlk)]);
    }
    for (int i = tid; i < kKp; i += kThreads) out[i] = -1;
    __syncthreads();
    auto pos_of = [&](int i) { return sh.kept[i / kBlk] * kBlk + i % kBlk; };
    if (n_cand <= kKp) {
        for (int i = tid; i < n_cand; i += kThreads) out[i] = pos_of(i);
    } else {
        // at least kKp positions reach the kKp-th best block's maximum (the kept
        // blocks' own maxima), so the kKp best all sit at or above it; the
        // candidates (at most 8 kKp) always fit the filter's capacity
        const int total = filter_ge(
            n_cand, thr2, [&](int i) { return sh.cand[i]; }, sh.cand2, sh.cand_idx, kMaxFiltered2, sh);
        select_top(
            total, kKp, [&](int i) { return sh.cand2[i]; },
            [&](uint32_t rank, int i) { out[rank] = pos_of(sh.cand_idx[i]); }, sh);
    }
    if (tid == 0 && n_sel_out) n_sel_out[b] = min(n_cand, kKp);
    trace_end(kTraceSelect);
}

}  // namespace

CSA2_TRACE_SETTER(trace_set_select)

cudaError_t preload_select() {
    const cudaError_t e = preload_kernel(k_select_topk<SelWide>, (int)sizeof(SelShared<SelWide>));
    return e != cudaSuccess ? e : preload_kernel(k_select_topk<SelHalf>, (int)sizeof(SelShared<SelHalf>));
}

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
    // loads the kernel and sets its shared-memory limit on this device, once per device
    if (const int rc = ensure_loaded()) return rc;
    // A small batch leaves most SMs idle with one CTA per sequence: then each
    // sequence's level-1 pass over its block maxima is spread over a cluster of
    // kClMax CTAs, when the grid stays within p->max_ctas (0: two waves of the SMs).
    // A batch of more sequences than SMs runs the 512-thread build, two CTAs per SM.
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return check_launch("select_topk: device");
    const int64_t cta_cap = p->max_ctas > 0 ? p->max_ctas : 2 * (int64_t)sms;
    const int ncl = (int64_t)B * kClMax <= cta_cap ? kClMax : 1;
    const bool half = ncl == 1 && B > sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * ncl));
    cfg.blockDim = dim3(half ? SelHalf::kThreads : SelWide::kThreads);
    cfg.dynamicSmemBytes = half ? (int)sizeof(SelShared<SelHalf>) : (int)sizeof(SelShared<SelWide>);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ncl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        half ? cudaLaunchKernelEx(&cfg, k_select_topk<SelHalf>, max_ncomp, p->compress_ratio, scores,
                                  block_max, n_tokens, idx, n_sel, dev_status, ncl)
             : cudaLaunchKernelEx(&cfg, k_select_topk<SelWide>, max_ncomp, p->compress_ratio, scores,
                                  block_max, n_tokens, idx, n_sel, dev_status, ncl);
    if (e != cudaSuccess) return check_launch("select_topk");
    return check_launch("select_topk");
}
