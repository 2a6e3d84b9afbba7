// Indexer for many queries against one key stream: the prefill chunk, where
// every query of the chunk scores the same sequence's index keys, up to its own
// causal length. "DeepSeek-V4.1-Flash-NVFP4" §3.3 (32 FP4 index heads, ReLU,
// per-head weights, sum; blocks of 8 positions scored by their best position);
// "CSA2稀疏注意力、384专家MoE与1M上下文" §2.1 (index_n_heads 32, index_head_dim 128).
//
// Here scoring is a dense contraction, so it runs as a block-scaled FP4 GEMM:
// four queries form one MMA's N = 4 x 32 heads = 128 rows of B, a 128-position
// key tile is A (the same tiled key cache the decode Indexer reads: 8 KB of E2M1
// codes with the 64-byte swizzle, 1 KB of E4M3 scales in scale-factor order), and
// D[128 x 128] = K . Q^T takes two tcgen05.mma.kind::mxf4nvf4 (K = 64 each). A
// persistent CTA walks a contiguous range of (query block of 16, key super-tile
// of 4 tiles) items: each 36 KB super-tile is loaded once per 16 queries. The
// epilogue is 16 warps, one per (TMEM lane quarter, query of the group): each reads
// its query's 32 head columns for 32 keys (one per lane), applies ReLU and the head
// weights in packed FP32 pairs, masks positions past the query's own causal
// length, and writes the score and the block maximum (8 adjacent lanes). Every
// wait is bounded.
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace csa2 {
namespace {
using namespace sm100;

constexpr int kKeyTile = CSA2_KEY_TILE;             // 128 positions
constexpr int kKeyTileBytes = CSA2_KEY_TILE_BYTES;  // 9216
constexpr int kKeyValBytes = kKeyTile * (kDi / 2);  // 8192
constexpr int kQPerGroup = 4;                       // queries per MMA
constexpr int kN = kQPerGroup * kHi;                // 128 = MMA N
constexpr int kGroups = 4;                          // MMA groups per query block
constexpr int kQPerBlock = kQPerGroup * kGroups;    // 16
constexpr int kTilesPerStage = 4;
constexpr int kStageBytes = kTilesPerStage * kKeyTileBytes;  // 36,864
constexpr int kPosPerStage = kTilesPerStage * kKeyTile;      // 512
constexpr int kStages = 4;
constexpr int kEpiWarps = 4 * kQPerGroup;           // 16: TMEM lane quarter x query of the group
constexpr int kAcc = 3;                             // accumulators in flight
constexpr int kLoadWarp = kEpiWarps, kMmaWarp = kLoadWarp + 1;
constexpr int kThreadsSh = 32 * (kMmaWarp + 1);     // 576
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 0;                       // kAcc x 128 columns
constexpr uint32_t kColSFA = kN * kAcc;             // 2 super-tile slots x kTilesPerStage x 8
constexpr uint32_t kColSFB = kColSFA + 2 * kTilesPerStage * 8;  // 2 query slots x kGroups x 8
static_assert(kColSFB + 2 * kGroups * 8 <= kTmemCols, "TMEM columns");
// kind::mxf4nvf4, A and B E2M1, K-major, dense, N = 128 (N>>3 in bits 17..22),
// UE4M3 scales, M = 128 (M>>4 in bits 24..28).
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) | ((128u >> 4) << 24);

struct ShShared {
    uint8_t stage[kStages][kStageBytes];  // key super-tiles (every stage 1024-aligned)
    uint8_t q[2][kGroups][kN * 64];       // B operand per group: 128 rows x 64 B, 64-byte swizzle
    uint8_t sfb[2][kGroups][1024];        // B scale factors per group, two 512-byte atoms
    float w[2][kQPerBlock][kHi];          // head weights of the block's queries
    int32_t nc[2][kQPerBlock];            // compressed length seen by each query (0 past Q)
    int32_t ncmax[2];                     // the block's longest
    uint64_t full[kStages], empty[kStages], qfull[2], qempty[2], accf[kAcc], acce[kAcc], done;
    uint32_t tmem_base;
    int abort;
};
constexpr int kShSmem = (int)sizeof(ShShared) + 1024;
// shared addresses stay below 256 KB, so a descriptor's 14-bit start-address field
// (address >> 4) can be advanced by adding (offset >> 4) without a carry out
static_assert(kShSmem <= 232448, "shared memory per block");

struct Work {
    int n_blocks;
    int64_t st_per_block;  // super-tiles of the longest query: the item grid is uniform
};

// tiles in super-tile g for a block whose longest query sees ncmax positions
__device__ __forceinline__ int tiles_in(int64_t g, int32_t ncmax) {
    const int64_t nt = (ncmax + kKeyTile - 1) / kKeyTile;
    const int64_t left = nt - g * kTilesPerStage;
    return left <= 0 ? 0 : (left < kTilesPerStage ? (int)left : kTilesPerStage);
}

// Packed FP32 pairs: fma.rn.f32x2 rounds each half exactly as fma.rn.f32 does, and
// one instruction covers two heads.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t v;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
    return v;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// sum over heads of w ReLU(d) (w2[i] = the weights of heads 2i, 2i + 1): ReLU as a
// max, the products and sums in packed pairs, eight independent partial sums. Every
// partial sum is exact when the products are (power-of-two scales), so the order of
// the chains does not change the result there.
__device__ __forceinline__ float head_sum(const uint64_t (&w2)[kHi / 2], const uint32_t (&r)[kHi]) {
    uint64_t c2[4] = {0ull, 0ull, 0ull, 0ull};  // +0.0f in both halves
#pragma unroll
    for (int h = 0; h < kHi; h += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float d0 = fmaxf(__uint_as_float(r[h + 2 * u]), 0.0f);
            const float d1 = fmaxf(__uint_as_float(r[h + 2 * u + 1]), 0.0f);
            c2[u] = fma2(w2[h / 2 + u], pack2(d0, d1), c2[u]);
        }
    }
    float v[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) unpack2(c2[u], v[2 * u], v[2 * u + 1]);
    return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

__global__ void __launch_bounds__(kThreadsSh, 1)
k_index_shared_tc(int Q, Work wk, int64_t max_ncomp, int ratio, const uint8_t* __restrict__ q_vals,
                  const uint8_t* __restrict__ q_scales, const float* __restrict__ w,
                  const uint8_t* __restrict__ keys, const int32_t* __restrict__ n_tokens,
                  float* scores, float* block_max, int32_t* dev_status) {
    extern __shared__ uint8_t smem_raw[];
    // aligned by offsetting the shared array itself, so that accesses through sh
    // stay shared-space loads and stores
    ShShared& sh = *reinterpret_cast<ShShared*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &sh.abort;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.qfull[i], 1);
            mbar_init(&sh.qempty[i], 1 + kEpiWarps);  // the MMA thread and every epilogue warp
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(&sh.accf[i], 1);
            mbar_init(&sh.acce[i], 32 * kEpiWarps);  // every epilogue thread
        }
        mbar_init(&sh.done, 1);
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const int64_t total = (int64_t)wk.n_blocks * wk.st_per_block;
    const int64_t f0 = total * blockIdx.x / gridDim.x;
    const int64_t f1 = total * (blockIdx.x + 1) / gridDim.x;
    const int64_t ld_bm = (max_ncomp + kBlk - 1) / kBlk;

    if (warp == kLoadWarp) {
        // ---------------- loader: the query block at each block change, super-tiles per stage
        int seg = -1, prev_k = -1;
        int64_t issued = 0;
        for (int64_t f = f0; f < f1; ++f) {
            const int k = (int)(f / wk.st_per_block);
            const int64_t g = f - (int64_t)k * wk.st_per_block;
            if (k != prev_k) {
                ++seg;
                const int qs = seg & 1;
                if (!mbar_wait_sleep(&sh.qempty[qs], ((seg >> 1) & 1) ^ 1, abort)) break;
                // row n = 32 qi + h of group gi: lane h copies head h of the 16 queries
                int32_t mx = 0;
#pragma unroll 4
                for (int qb = 0; qb < kQPerBlock; ++qb) {
                    const int qq = k * kQPerBlock + qb;
                    const int gi = qb / kQPerGroup, n = kHi * (qb % kQPerGroup) + lane;
                    uint8_t* row = sh.q[qs][gi] + n * 64;
                    uint4 v[4] = {};
                    uint2 sc = make_uint2(0u, 0u);
                    int32_t nc = 0;
                    float wv = 0.f;
                    if (qq < Q) {
                        const uint4* src = reinterpret_cast<const uint4*>(q_vals + ((int64_t)qq * kHi + lane) * (kDi / 2));
#pragma unroll
                        for (int c = 0; c < 4; ++c) v[c] = src[c];
                        sc = *reinterpret_cast<const uint2*>(q_scales + ((int64_t)qq * kHi + lane) * (kDi / 16));
                        wv = w[(int64_t)qq * kHi + lane];
                        int64_t n_c = n_tokens[qq] / ratio;
                        if (n_c > max_ncomp || n_c < 0) {
                            if (lane == 0) raise_status(dev_status, CSA2_DEV_BAD_LENGTH);
                            n_c = n_c < 0 ? 0 : max_ncomp;
                        }
                        nc = (int32_t)n_c;
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(row + ((c ^ ((n >> 1) & 3)) << 4)) = v[c];
                    // scale-factor atoms: row n & 31 = h, bytes 4 qi .. 4 qi + 3
                    *reinterpret_cast<uint32_t*>(&sh.sfb[qs][gi][lane * 16 + 4 * (qb % kQPerGroup)]) = sc.x;
                    *reinterpret_cast<uint32_t*>(&sh.sfb[qs][gi][512 + lane * 16 + 4 * (qb % kQPerGroup)]) = sc.y;
                    sh.w[qs][qb][lane] = wv;
                    if (lane == 0) sh.nc[qs][qb] = nc;
                    mx = max(mx, nc);
                }
                if (lane == 0) sh.ncmax[qs] = mx;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.qfull[qs]);
                prev_k = k;
            }
            const int qs = seg & 1;
            // every lane reads the block's length after its own writes above
            const int nt = tiles_in(g, sh.ncmax[qs]);
            if (nt == 0) continue;  // past this block's longest query: nothing to load
            const int64_t i = issued;
            const int s = (int)(i % kStages);
            if (!mbar_wait_sleep(&sh.empty[s], (uint32_t)((i / kStages) & 1) ^ 1, abort)) break;
            if (lane == 0) {
                const uint32_t bytes = (uint32_t)nt * kKeyTileBytes;
                mbar_arrive_expect_tx(&sh.full[s], bytes);
                bulk_g2s(sh.stage[s], keys + g * kStageBytes, bytes, &sh.full[s]);
            }
            __syncwarp();
            issued = i + 1;
        }
        // copies still in flight land before the CTA can exit
        for (int64_t j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
            for (uint32_t k2 = 0; k2 < kSpinLimit; ++k2)
                if (mbar_try_wait(&sh.full[j % kStages], (uint32_t)((j / kStages) & 1))) break;
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer: the whole warp runs the loop (its values stay
        // warp-uniform) and waits; one elected lane issues every copy, MMA and commit.
        // Per tile two scale copies, then per query group two MMAs into the next
        // accumulator.
        const bool leader = elect_one();
        int seg = -1, prev_k = -1;
        int s = 0, a = 0;             // stage and accumulator slots
        uint32_t sph = 0, aph = 0;    // their phase parities
        const uint32_t full0 = smem_u32(&sh.full[0]), empty0 = smem_u32(&sh.empty[0]);
        const uint32_t accf0 = smem_u32(&sh.accf[0]), acce0 = smem_u32(&sh.acce[0]);
        const uint32_t stage0 = smem_u32(sh.stage[0]);
        const uint64_t dA0 = smem_desc(stage0, 16, 512, kLayoutSw64);
        const uint64_t dB0 = smem_desc(smem_u32(sh.q[0][0]), 16, 512, kLayoutSw64);
        int tile_par = 0;
        bool ok = true;
        int k = (int)(f0 / wk.st_per_block);
        int g = (int)(f0 - (int64_t)k * wk.st_per_block);
        const int spb = (int)wk.st_per_block;
        for (int left = (int)(f1 - f0); left > 0 && ok; --left, g = (g + 1 == spb) ? (++k, 0) : g + 1) {
            if (k != prev_k) {
                if (seg >= 0 && leader) tc_commit(&sh.qempty[seg & 1]);
                ++seg;
                const int qs = seg & 1;
                if (!mbar_wait_sleep(&sh.qfull[qs], (uint32_t)((seg >> 1) & 1), abort)) break;
                tc_fence_after();
                if (leader) {
                    for (int gi = 0; gi < kGroups; ++gi) {
                        const uint32_t sfb = smem_u32(sh.sfb[qs][gi]);
                        const uint32_t col = tmem + kColSFB + 32 * qs + 8 * gi;
                        tmem_cp_32x128b_x4(col, smem_desc(sfb, 128, 128, kLayoutNone));
                        tmem_cp_32x128b_x4(col + 4, smem_desc(sfb + 512, 128, 128, kLayoutNone));
                    }
                }
                __syncwarp();
                prev_k = k;
            }
            const int qs = seg & 1;
            const int nt = tiles_in(g, sh.ncmax[qs]);
            if (nt == 0) continue;
            if (!mbar_wait_sleep_at(full0 + 8u * s, sph, abort)) break;
            tc_fence_after();
            // the key scales of every tile of the super-tile, in the slot of this
            // super-tile's parity: the other slot may still feed the previous one
            const uint32_t sfa0 = tmem + kColSFA + 8 * kTilesPerStage * tile_par;
            tile_par ^= 1;
            const uint32_t st0 = stage0 + (uint32_t)s * kStageBytes;
            if (leader) {
                for (int j = 0; j < nt; ++j) {
                    const uint32_t sf = st0 + j * kKeyTileBytes + kKeyValBytes;
                    tmem_cp_32x128b_x4(sfa0 + 8 * j, smem_desc(sf, 128, 128, kLayoutNone));
                    tmem_cp_32x128b_x4(sfa0 + 8 * j + 4, smem_desc(sf + 512, 128, 128, kLayoutNone));
                }
            }
            __syncwarp();
            // group-major: the epilogue keeps one query's weights across the tiles.
            // Descriptors advance by (byte offset >> 4) in their start-address field.
            const uint64_t dA_s = dA0 + (uint64_t)(((uint32_t)s * kStageBytes) >> 4);
            for (int gi = 0; gi < kGroups && ok; ++gi) {
                const uint64_t dB = dB0 + (uint64_t)(((uint32_t)(qs * kGroups + gi) * (kN * 64)) >> 4);
                const uint32_t sfb = tmem + kColSFB + 32 * qs + 8 * gi;
                uint64_t dA = dA_s;
                uint32_t sfa = sfa0;
                for (int j = 0; j < nt; ++j, dA += kKeyTileBytes >> 4, sfa += 8) {
                    if (!mbar_wait_sleep_at(acce0 + 8u * a, aph ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (leader) {
                        const uint32_t d = tmem + kColD + kN * a;
                        mma_mxf4nvf4(d, dA, dB, kIdesc, sfa, sfb, 0);
                        mma_mxf4nvf4(d, dA + 2, dB + 2, kIdesc, sfa + 4, sfb + 4, 1);  // K 64..127
                        tc_commit_at(accf0 + 8u * a);
                    }
                    __syncwarp();
                    a = (a + 1 == kAcc) ? 0 : a + 1;
                    aph ^= (a == 0) ? 1u : 0u;
                }
            }
            if (leader) tc_commit_at(empty0 + 8u * s);
            __syncwarp();
            if (++s == kStages) {
                s = 0;
                sph ^= 1u;
            }
        }
        if (leader) {
            if (seg >= 0) tc_commit(&sh.qempty[seg & 1]);
            // every MMA and copy issued above has completed before TMEM is freed
            tc_commit(&sh.done);
        }
        __syncwarp();
        for (uint32_t k2 = 0; k2 < kSpinLimit; ++k2)
            if (mbar_try_wait(&sh.done, 0)) break;
    } else {
        // ---------------- epilogue: warp (qp, wq) reads TMEM lanes 32 wq.. (positions
        // 32 wq.. of each tile) and the 32 columns of query qp of the item's group; it
        // releases the accumulator as soon as its columns are in registers.
        const int wq = warp & 3, qp = warp >> 2;
        const uint32_t accf0 = smem_u32(&sh.accf[0]), acce0 = smem_u32(&sh.acce[0]);
        const uint32_t tmem_lane = tmem + ((uint32_t)(32 * wq) << 16) + kColD + kHi * qp;
        const bool blk_lead = (lane & (kBlk - 1)) == 0;
        int seg = -1, prev_k = -1;
        int a = 0;         // accumulator slot of the next item
        uint32_t ph = 0;   // its phase parity
        bool ok = true;
        int k = (int)(f0 / wk.st_per_block);
        int g = (int)(f0 - (int64_t)k * wk.st_per_block);
        const int spb = (int)wk.st_per_block;
        for (int left = (int)(f1 - f0); left > 0 && ok; --left, g = (g + 1 == spb) ? (++k, 0) : g + 1) {
            if (k != prev_k) {
                if (seg >= 0) {  // done with the previous block's weights and lengths
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.qempty[seg & 1]);
                }
                ++seg;
                if (!mbar_wait_sleep(&sh.qfull[seg & 1], (uint32_t)((seg >> 1) & 1), abort)) break;
                prev_k = k;
            }
            const int qs = seg & 1;
            const int nt = tiles_in(g, sh.ncmax[qs]);
            // group-major, as the MMA issuer runs: the query's weights stay in registers
            // across the super-tile's tiles
            for (int gi = 0; gi < kGroups && ok; ++gi) {
                const int qb = gi * kQPerGroup + qp;  // this warp's query of group gi
                const int32_t nc0 = sh.nc[qs][qb];
                const int64_t qq = (int64_t)(k * kQPerBlock + qb);
                float* srow0 = scores + qq * max_ncomp;
                float* brow0 = block_max + qq * ld_bm;
                uint64_t w0[kHi / 2];
#pragma unroll
                for (int h4 = 0; h4 < kHi / 4; ++h4) {
                    const ulonglong2 v0 = reinterpret_cast<const ulonglong2*>(sh.w[qs][qb])[h4];
                    w0[2 * h4] = v0.x, w0[2 * h4 + 1] = v0.y;
                }
                int tl = g * kPosPerStage + 32 * wq + lane;  // this lane's position in tile j
                float* sp = srow0 + tl;  // its score and block-maximum slots, stepped per tile
                float* bp = brow0 + (tl >> 3);
                for (int j = 0; j < nt; ++j, tl += kKeyTile, sp += kKeyTile, bp += kKeyTile / kBlk) {
                    if (!mbar_wait_sleep_at(accf0 + 8u * a, ph, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t r[kHi];
                    tmem_ld_32x32b_x32_nowait(tmem_lane + kN * a, r);
                    tmem_wait_ld_regs32(r);
                    tc_fence_before();
                    mbar_arrive_at(acce0 + 8u * a);  // this thread's part of the accumulator is read
                    a = (a + 1 == kAcc) ? 0 : a + 1;
                    ph ^= (a == 0) ? 1u : 0u;
                    const float sc = head_sum(w0, r);
                    const bool v = tl < nc0;
                    float m = v ? sc : -INFINITY;
#pragma unroll
                    for (int o = 1; o < kBlk; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    st_global_if(sp, sc, v);
                    st_global_if(bp, m, v && blk_lead);
                }
            }
        }
        if (ok && seg >= 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.qempty[seg & 1]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && sh.abort) raise_status(dev_status, CSA2_DEV_TIMEOUT);
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int sm_count_sh() {
    static int n[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    if (!n[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        n[dev] = v > 0 ? v : 1;
    }
    return n[dev];
}

}  // namespace

cudaError_t preload_index_shared() { return preload_kernel(k_index_shared_tc, kShSmem); }

}  // namespace csa2

using namespace csa2;

extern "C" int csa2_index_scores_shared(const csa2_params* p, int Q, int64_t max_ncomp,
                                        const uint8_t* q_vals,
                                        const uint8_t* q_scales, const float* w,
                                        const uint8_t* key_cache, const int32_t* n_tokens,
                                        float* scores, float* block_max, int32_t* dev_status,
                                        void* stream) {
    CSA2_CHECK_PARAMS(p);
    if (Q < 0 || max_ncomp < 0)
        return fail(CSA2_ERR_INVALID_ARG, "index_scores_shared: negative size");
    if (p->index_heads != kHi || p->index_dim != kDi || p->block_size != kBlk || p->compress_ratio < 1)
        return fail(CSA2_ERR_UNSUPPORTED, "index_scores_shared: built for 32 heads x 128, blocks of 8");
    if (max_ncomp > (int64_t)INT32_MAX - kPosPerStage)
        return fail(CSA2_ERR_UNSUPPORTED, "index_scores_shared: positions are 32-bit in the kernel");
    if (Q == 0 || max_ncomp == 0) return CSA2_OK;
    if (!q_vals || !q_scales || !w || !key_cache || !n_tokens || !scores || !block_max)
        return fail(CSA2_ERR_INVALID_ARG, "index_scores_shared: NULL buffer");
    if (!aligned16(q_vals) || !aligned16(key_cache) || (reinterpret_cast<uintptr_t>(q_scales) & 7) ||
        (reinterpret_cast<uintptr_t>(w) & 3))
        return fail(CSA2_ERR_ALIGN, "index_scores_shared: q_vals, key_cache 16-byte, q_scales 8-byte aligned");
    // loads the kernel and sets its shared-memory limit on this device, once per device
    if (const int rc = ensure_loaded()) return rc;
    Work wk;
    wk.n_blocks = (Q + kQPerBlock - 1) / kQPerBlock;
    wk.st_per_block = (max_ncomp + kPosPerStage - 1) / kPosPerStage;
    const int64_t items = (int64_t)wk.n_blocks * wk.st_per_block;
    int64_t ctas = sm_count_sh();
    if (p->max_ctas > 0 && p->max_ctas < ctas) ctas = p->max_ctas;
    const int grid = (int)(items < ctas ? items : ctas);
    k_index_shared_tc<<<grid, kThreadsSh, kShSmem, static_cast<cudaStream_t>(stream)>>>(
        Q, wk, max_ncomp, p->compress_ratio, q_vals, q_scales, w, key_cache, n_tokens, scores,
        block_max, dev_status);
    return check_launch("index_scores_shared");
}
