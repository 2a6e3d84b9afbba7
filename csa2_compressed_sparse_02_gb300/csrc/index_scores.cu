// Decode Indexer with fused block maximum, and the writer of its key cache.
// "DeepSeek-V4.1-Flash-NVFP4" §3.3: 32 FP4 index query heads score the shared
// FP4 index key; ReLU, per-head weights, sum; blocks of 8 positions are scored
// by their best position.
//
// Key cache: tiles of 128 positions, each the 9216-byte shared-memory image the
// tensor cores read (8 KB of E2M1 codes, K-major with the 64-byte swizzle, then
// 1 KB of E4M3 group scales in the scale-factor order of block-scaled MMA; the
// exact formulas are in include/csa2.h). One bulk copy moves one tile.
//
// Tensor-core build (k_index_scores_tc): per 128-position tile, D[128 x 32] =
// K[128 x 128] . Q[32 x 128]^T as two tcgen05 block-scaled FP4 MMAs (K = 64 each,
// UE4M3 scale per 16 elements) into TMEM; the epilogue warps read one position
// per lane (32 heads), apply ReLU and the head weights, and reduce the block
// maximum over 8 adjacent lanes. One persistent CTA per SM; warps 0-7 epilogue
// (two warpgroups taking alternate super-tiles), warp 8 loads (one bulk copy
// per super-tile of 6 tiles into a 4-stage ring), warps 9 and 10 issue the
// MMAs of alternate super-tiles (a single issuing thread serialises each scale
// copy with its MMA; two overlap them), each into its own TMEM accumulators.
//
// CUDA-core build (k_index_scores_cc): one thread per position, 32 fp32
// accumulators, the query decoded once per CTA into shared memory.
#include "common.cuh"
#include "sm100.cuh"

#include <algorithm>

namespace csa2 {
namespace {

constexpr int kKeyTile = CSA2_KEY_TILE;            // 128 positions
constexpr int kKeyTileBytes = CSA2_KEY_TILE_BYTES;  // 9216
constexpr int kKeyValBytes = kKeyTile * (kDi / 2);  // 8192

// byte offset, inside a tile, of 16-byte chunk c (dims 32c..32c+31) of position m
__device__ __forceinline__ int key_val_off(int m, int c) { return m * 64 + ((c ^ ((m >> 1) & 3)) << 4); }
// byte offset, inside a tile, of the 4 scales of groups 4h..4h+3 of position m
__device__ __forceinline__ int key_scale_off(int m, int h) {
    return kKeyValBytes + h * 512 + (m & 31) * 16 + (m >> 5) * 4;
}

__device__ __forceinline__ int64_t seq_ncomp(const int32_t* n_tokens, int b, int ratio,
                                            int64_t max_ncomp, int32_t* dev_status, bool report) {
    int64_t n_c = n_tokens[b] / ratio;
    if (n_c > max_ncomp || n_c < 0) {
        if (report) raise_status(dev_status, CSA2_DEV_BAD_LENGTH);
        n_c = n_c < 0 ? 0 : max_ncomp;
    }
    return n_c;
}

// ------------------------------------------------------------------ key writer
__global__ void __launch_bounds__(256)
k_index_keys_write(int B, int64_t n, const uint8_t* __restrict__ vals,
                   const uint8_t* __restrict__ scales, const int64_t* __restrict__ pos0,
                   uint8_t* const* dst, const int64_t* __restrict__ cap, int32_t* dev_status) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (int64_t)B * n) return;
    const int b = (int)(e / n);
    const int64_t t = pos0[b] + (e - (int64_t)b * n);
    if (t < 0 || t >= cap[b]) {
        raise_status(dev_status, CSA2_DEV_BAD_LENGTH);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(vals + e * (kDi / 2));
    uint8_t* tile = dst[b] + (t / kKeyTile) * kKeyTileBytes;
    const int m = (int)(t % kKeyTile);
#pragma unroll
    for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(tile + key_val_off(m, c)) = src[c];
    const uint2 sc = *reinterpret_cast<const uint2*>(scales + e * (kDi / kGroup));
    *reinterpret_cast<uint32_t*>(tile + key_scale_off(m, 0)) = sc.x;
    *reinterpret_cast<uint32_t*>(tile + key_scale_off(m, 1)) = sc.y;
}

// ------------------------------------------------------------------ CUDA-core build
constexpr int kKeysPerCta = 256;

__global__ void __launch_bounds__(kKeysPerCta)
k_index_scores_cc(int64_t max_ncomp, int ratio, const uint8_t* __restrict__ q_vals,
                  const uint8_t* __restrict__ q_scales, const float* __restrict__ w,
                  const uint8_t* const* key_cache, const int32_t* __restrict__ n_tokens,
                  float* scores, float* block_max, int32_t* dev_status) {
    __shared__ float4 sq[kDi][kHi / 4];  // sq[d][h/4] = q[h..h+3][d]
    __shared__ float sw[kHi];
    const int b = blockIdx.y, tid = threadIdx.x;
    const int64_t n_c = seq_ncomp(n_tokens, b, ratio, max_ncomp, dev_status,
                                  tid == 0 && blockIdx.x == 0);
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
        const uint8_t* tile = key_cache[b] + (t / kKeyTile) * kKeyTileBytes;
        const int m = (int)(t % kKeyTile);
        const uint32_t sc[2] = {*reinterpret_cast<const uint32_t*>(tile + key_scale_off(m, 0)),
                                *reinterpret_cast<const uint32_t*>(tile + key_scale_off(m, 1))};
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {  // 16 bytes = 32 dims = 2 groups
            const uint4 kb = *reinterpret_cast<const uint4*>(tile + key_val_off(m, q4));
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
    float mx = valid ? s : -INFINITY;
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    if (valid && (tid & (kBlk - 1)) == 0)
        block_max[(int64_t)b * ((max_ncomp + kBlk - 1) / kBlk) + t / kBlk] = mx;
}

// ------------------------------------------------------------------ tensor-core build
// Unit of work: a super-tile of up to kTilesPerStage consecutive tiles of one sequence
// (contiguous in the cache, so one bulk copy of up to 54 KB). Per super-tile the
// MMA thread issues 2 scale copies + 2 MMAs per tile into the tile's own TMEM
// accumulator, then one commit for the stage and one for the epilogue: the
// fixed per-commit, per-copy and per-handoff costs are paid once per 54 KB, not
// per 9 KB. Those costs, not the bytes in flight, set the rate: at 1 M context
// (1.28 GB per launch) super-tiles of 2 / 3 / 4 / 5 tiles in 10 / 7 / 5 / 4
// stages took 0.256 / 0.227 / 0.205 / 0.203 ms, and 6 tiles in 4 stages the same
// as 5. Six tiles fill the TMEM (2 x 6 x 32 accumulator columns, 2 x 6 x 8 scale
// columns, 32 query scale columns), and a ring of four such stages fits in shared
// memory because no per-sequence table is kept there.
constexpr int kTilesPerStage = 6;
constexpr int kStageBytes = kTilesPerStage * kKeyTileBytes;  // 55,296 = 54 x 1024
constexpr int kStages = 4;
constexpr int kIssuers = 2;      // MMA-issuing warps, alternating super-tiles
// Each issuer waits only for the stage fills of its own super-tiles. A parity
// wait is exact only if the phase before the awaited one has completed, i.e.
// the waiter saw the stage's previous fill itself: so every use of a stage must
// belong to the same issuer, which needs kStages to be a multiple of kIssuers.
// With an odd ring a stage alternates between the issuers, and an issuer whose
// previous fill of that stage (the other issuer's copy) was still in flight
// read the preceding phase as the awaited one and went ahead on a stage being
// filled; its commit then freed the stage once too often.
static_assert(kStages % kIssuers == 0, "every use of a stage must belong to one issuer");
constexpr int kAcc = kIssuers;   // one super-tile accumulator set per issuer
constexpr int kEpiGroups = 2;    // epilogue warpgroups, alternating super-tiles
constexpr int kLoadWarp = 4 * kEpiGroups, kMmaWarp = kLoadWarp + 1;
constexpr int kTcThreads = 32 * (kMmaWarp + kIssuers);  // 0-7 epilogue, 8 loader, 9-10 MMA
constexpr uint32_t kTmemCols = 512;
// TMEM columns: D[kAcc][kTilesPerStage] x 32, SFA[kAcc][kTilesPerStage] x 8, SFB[kIssuers][2] x 8
constexpr uint32_t kColD = 0, kColSFA = 32 * kAcc * kTilesPerStage, kColSFB = kColSFA + 8 * kAcc * kTilesPerStage;
static_assert(kColSFB + 16 * kIssuers <= kTmemCols, "TMEM columns");
// Instruction descriptor: kind::mxf4nvf4, A and B E2M1 (1), K-major, dense,
// N = 32 (N>>3 in bits 17..22), UE4M3 scales (bit 23 = 0), M = 128 (M>>4 in bits 24..28).
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

struct TcShared {
    uint8_t stage[kStages][kStageBytes];  // every stage 1024-aligned
    uint8_t q[2][kHi * (kDi / 2)];         // B operand (32 heads x 64 B, 64-byte swizzle), 2 slots
    uint8_t sfb[2][1024];                  // B scale factors, two 512-byte atoms per slot
    uint64_t full[kStages], empty[kStages];
    uint64_t qfull[2], qempty[2], accf[kAcc], acce[kAcc], done;
    int64_t total;  // super-tiles of all sequences
    uint32_t tmem_base;
    int abort;
};

// super-tiles of a sequence with n_c positions
__device__ __forceinline__ int64_t supers_of(int64_t n_c) {
    return (n_c + kTilesPerStage * kKeyTile - 1) / (kTilesPerStage * kKeyTile);
}

// The sequence of each flat super-tile (super-tiles numbered sequence after
// sequence) for a role that visits increasing f: it reads each sequence's length
// as it passes it, so no per-sequence table sits in shared memory and the batch
// size is not bounded by it. f must be below the total.
// Every role of every CTA must read the same n_tokens values that warp 0 summed
// into the total: the loader, the MMA issuers and the epilogue each walk the
// flat super-tiles with their own cursor, and a role that saw other lengths
// would wait on barriers the others never complete (until the bounded wait
// gives up). That holds because n_tokens does not change while the kernel runs:
// the kernel is launched programmatically behind the Compressor (which writes
// n_tokens), so its CTAs may be placed and set up their barriers and TMEM while
// that kernel still runs, but nothing global is read before grid_dep_wait(),
// i.e. before the kernels ahead of it on the stream have completed.
struct SeqCursor {
    int b = -1;
    int64_t start = 0, end = 0;  // flat super-tiles [start, end) belong to sequence b
    int64_t n_c = 0;
    __device__ __forceinline__ void advance(int64_t f, const int32_t* n_tokens, int ratio,
                                            int64_t max_ncomp) {
        while (f >= end) {
            ++b;
            start = end;
            n_c = seq_ncomp(n_tokens, b, ratio, max_ncomp, nullptr, false);
            end = start + supers_of(n_c);
        }
    }
};

// The super-tiles of one CTA, in increasing order: chunks of kChunk super-tiles
// (442 KB) dealt round robin over the grid, then the remainder cut into equal
// contiguous ranges. At any moment the CTAs stream neighbouring chunks of the
// cache, which spreads the load over the memory system more evenly than one
// long contiguous range per CTA (whose end times spread by tens of microseconds
// in a read of the same size); a chunk is long enough that sequence changes
// (each a new query slot, two slots deep) stay rare against the stage ring.
constexpr int kChunk = 8;
struct TileIter {
    int64_t f, end, total, body;
    int k, rounds;
    __device__ __forceinline__ void init(int64_t total_) {
        total = total_;
        rounds = (int)(total / kChunk / gridDim.x);
        body = (int64_t)rounds * gridDim.x * kChunk;
        k = 0;
        set();
    }
    __device__ __forceinline__ void set() {
        if (k < rounds) {
            f = ((int64_t)k * gridDim.x + blockIdx.x) * kChunk;
            end = f + kChunk;
        } else {
            const int64_t rest = total - body;
            f = body + rest * blockIdx.x / gridDim.x;
            end = body + rest * (blockIdx.x + 1) / gridDim.x;
        }
    }
    // the next super-tile (flat index over all sequences); false when done
    __device__ __forceinline__ bool next(int64_t& out) {
        while (f >= end) {
            if (k >= rounds) return false;
            ++k;
            set();
        }
        out = f++;
        return true;
    }
};

// tiles in super-tile g of a sequence with n_c positions
__device__ __forceinline__ int tiles_in(int64_t g, int64_t n_c) {
    const int64_t nt = (n_c + kKeyTile - 1) / kKeyTile;
    const int64_t left = nt - g * kTilesPerStage;
    return left < kTilesPerStage ? (int)left : kTilesPerStage;
}

__global__ void __launch_bounds__(kTcThreads, 1)
k_index_scores_tc(int B, int64_t max_ncomp, int ratio, const uint8_t* __restrict__ q_vals,
                  const uint8_t* __restrict__ q_scales, const float* __restrict__ w,
                  const uint8_t* const* key_cache, const int32_t* __restrict__ n_tokens,
                  float* scores, float* block_max, int32_t* dev_status) {
    using namespace sm100;
    extern __shared__ uint8_t smem_raw[];
    // aligned by offsetting the shared array itself, so that accesses through sh
    // stay shared-space loads and stores
    TcShared& sh = *reinterpret_cast<TcShared*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &sh.abort;
    trace_start(kTraceIndex);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.qfull[i], 1);
            mbar_init(&sh.qempty[i], kIssuers);
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(&sh.accf[i], 1);
            mbar_init(&sh.acce[i], 4);
        }
        mbar_init(&sh.done, kIssuers);
        sh.abort = 0;
        fence_mbar_init();
    }
    // launched programmatically: nothing global is read before the kernels ahead of
    // it on the stream (the Compressor writes the lengths) have completed
    grid_dep_wait();
    if (warp == 0) {  // super-tiles of all sequences (CTA 0 flags bad lengths)
        int64_t local = 0;
        for (int b = lane; b < B; b += 32)
            local += supers_of(seq_ncomp(n_tokens, b, ratio, max_ncomp, dev_status, blockIdx.x == 0));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
        if (lane == 0) sh.total = local;
    }
    if (warp == kMmaWarp) {  // the first MMA warp owns the TMEM allocation
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const int64_t total = sh.total;
    TileIter ti;
    ti.init(total);

    if (warp == kLoadWarp) {
        // ---------------- loader: query slots per sequence, super-tiles per stage
        int seg = -1, b = 0, prev_b = -1;
        SeqCursor cur;
        int64_t issued = 0;
        // the key stream (72 B per position, far larger than L2) is read once: its
        // lines go first, so the scores and block maxima written here are still in
        // L2 when the selection reads them
        const uint64_t key_policy = l2_policy_evict_first();
        int64_t f, i = 0;
        for (; ti.next(f); ++i) {
            cur.advance(f, n_tokens, ratio, max_ncomp);
            b = cur.b;
            const int64_t g = f - cur.start;
            // the key copy first: it does not need the query, whose staging costs a
            // memory round trip at every sequence change
            const int s = (int)(i % kStages);
            if (!mbar_wait(&sh.empty[s], (uint32_t)((i / kStages) & 1) ^ 1, abort)) break;
            if (lane == 0) {
                const uint32_t bytes = (uint32_t)tiles_in(g, cur.n_c) * kKeyTileBytes;
                mbar_arrive_expect_tx(&sh.full[s], bytes);
                bulk_g2s_hint(sh.stage[s], key_cache[b] + g * kStageBytes, bytes, &sh.full[s],
                              key_policy);
            }
            __syncwarp();
            issued = i + 1;
            if (b != prev_b) {
                ++seg;
                const int qs = seg & 1;
                if (!mbar_wait(&sh.qempty[qs], ((seg >> 1) & 1) ^ 1, abort)) break;
                // lane h writes head h: 64 B of codes in the swizzled K-major image,
                // its 8 scales into the two scale-factor atoms (row h, bytes 0..3)
                const uint4* src = reinterpret_cast<const uint4*>(
                    q_vals + ((int64_t)b * kHi + lane) * (kDi / 2));
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(&sh.q[qs][lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)]) = src[c];
                const uint2 sc = *reinterpret_cast<const uint2*>(
                    q_scales + ((int64_t)b * kHi + lane) * (kDi / 16));
                *reinterpret_cast<uint4*>(&sh.sfb[qs][lane * 16]) = make_uint4(sc.x, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(&sh.sfb[qs][512 + lane * 16]) = make_uint4(sc.y, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.qfull[qs]);
                prev_b = b;
            }
        }
        // copies still in flight land before the CTA can exit
        for (int64_t j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
            for (uint32_t k = 0; k < kSpinLimit; ++k)
                if (mbar_try_wait(&sh.full[j % kStages], (uint32_t)((j / kStages) & 1))) break;
        }
    } else if (warp >= kMmaWarp) {
        // ---------------- MMA issuers: warp kMmaWarp + e issues super-tiles i with
        // i % kIssuers == e (a single thread each); every issuer copies the query
        // scale factors of every sequence segment into its own TMEM slots.
        const int e = warp - kMmaWarp;
        // descriptors built once; a stage, a tile or a query slot moves the start-address field
        const uint64_t dA0 = smem_desc(smem_u32(sh.stage[0]), 16, 512, kLayoutSw64);
        const uint64_t dS0 = smem_desc(smem_u32(sh.stage[0]) + kKeyValBytes, 128, 128, kLayoutNone);
        const uint64_t dQ0 = smem_desc(smem_u32(sh.q[0]), 16, 512, kLayoutSw64);
        if (lane == 0) {
            int seg = -1, b = 0, prev_b = -1;
            SeqCursor cur;
            int64_t f, i = 0;
            for (; ti.next(f); ++i) {
                cur.advance(f, n_tokens, ratio, max_ncomp);
                b = cur.b;
                if (b != prev_b) {
                    if (seg >= 0) tc_commit(&sh.qempty[seg & 1]);
                    ++seg;
                    const int qs = seg & 1;
                    if (!mbar_wait(&sh.qfull[qs], (uint32_t)((seg >> 1) & 1), abort)) break;
                    tc_fence_after();
                    const uint32_t sfb = smem_u32(sh.sfb[qs]);
                    const uint32_t col = tmem + kColSFB + 16 * e + 8 * qs;
                    tmem_cp_32x128b_x4(col, smem_desc(sfb, 128, 128, kLayoutNone));
                    tmem_cp_32x128b_x4(col + 4, smem_desc(sfb + 512, 128, 128, kLayoutNone));
                    prev_b = b;
                }
                if ((int)(i % kIssuers) != e) continue;
                const int s = (int)(i % kStages), a = (int)(i % kAcc);
                if (!mbar_wait(&sh.full[s], (uint32_t)((i / kStages) & 1), abort)) break;
                if (!mbar_wait(&sh.acce[a], (uint32_t)((i / kAcc) & 1) ^ 1, abort)) break;
                tc_fence_after();
                const int qs = seg & 1;
                const uint32_t sfb = tmem + kColSFB + 16 * e + 8 * qs;
                const int nt = tiles_in(f - cur.start, cur.n_c);
                // descriptors advance by (byte offset >> 4) in their start-address field
                // (shared addresses stay below 256 KB: no carry out of the field)
                const uint64_t dQ = dQ0 + (uint64_t)((uint32_t)(qs * kHi * (kDi / 2)) >> 4);
                uint64_t dA = dA0 + (uint64_t)((uint32_t)(s * kStageBytes) >> 4);
                uint64_t dS = dS0 + (uint64_t)((uint32_t)(s * kStageBytes) >> 4);
                uint32_t sfa = tmem + kColSFA + 8 * (a * kTilesPerStage);
                uint32_t d = tmem + kColD + 32 * (a * kTilesPerStage);
                for (int j = 0; j < nt; ++j, dA += kKeyTileBytes >> 4, dS += kKeyTileBytes >> 4, sfa += 8, d += 32) {
                    tmem_cp_32x128b_x4(sfa, dS);
                    tmem_cp_32x128b_x4(sfa + 4, dS + (512 >> 4));
                    mma_mxf4nvf4(d, dA, dQ, kIdesc, sfa, sfb, 0);
                    mma_mxf4nvf4(d, dA + 2, dQ + 2, kIdesc, sfa + 4, sfb + 4, 1);  // K 64..127
                }
                tc_commit(&sh.empty[s]);
                tc_commit(&sh.accf[a]);
            }
            // every MMA and copy issued above has completed before TMEM is freed
            tc_commit(&sh.done);
            for (uint32_t k = 0; k < kSpinLimit; ++k)
                if (mbar_try_wait(&sh.done, 0)) break;
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warpgroup e handles super-tiles i with i % kEpiGroups == e;
        // warp q of it owns TMEM lanes 32q..32q+31 = positions 32q.. of each tile
        const int eg = warp >> 2, wq = warp & 3;
        const int64_t ld_bm = (max_ncomp + kBlk - 1) / kBlk;
        int b = 0, prev_b = -1;
        SeqCursor cur;
        float wv[kHi];
        int64_t f, i = 0;
        for (; ti.next(f); ++i) {
            cur.advance(f, n_tokens, ratio, max_ncomp);
            b = cur.b;
            const int a = (int)(i % kAcc);
            if (b != prev_b) {
                const float4* w4 = reinterpret_cast<const float4*>(w + (int64_t)b * kHi);
#pragma unroll
                for (int h4 = 0; h4 < kHi / 4; ++h4) {
                    const float4 v = w4[h4];
                    wv[4 * h4] = v.x;
                    wv[4 * h4 + 1] = v.y;
                    wv[4 * h4 + 2] = v.z;
                    wv[4 * h4 + 3] = v.w;
                }
                prev_b = b;
            }
            if ((int)(i % kEpiGroups) != eg) continue;
            if (!mbar_wait(&sh.accf[a], (uint32_t)((i / kAcc) & 1), abort)) break;
            tc_fence_after();
            const int64_t g = f - cur.start;
            const int nt = tiles_in(g, cur.n_c);
            const int64_t n_c = cur.n_c;
            for (int j = 0; j < nt; ++j) {
                uint32_t r[kHi];
                tmem_ld_32x32b_x32(
                    tmem + ((uint32_t)(32 * wq) << 16) + kColD + 32 * (a * kTilesPerStage + j), r);
                float s = 0.0f;
#pragma unroll
                for (int h = 0; h < kHi; ++h) {
                    const float dh = __uint_as_float(r[h]);
                    s = __fmaf_rn(wv[h], dh > 0.0f ? dh : 0.0f, s);
                }
                const int64_t t = (g * kTilesPerStage + j) * kKeyTile + 32 * wq + lane;
                const bool valid = t < n_c;
                if (valid) scores[(int64_t)b * max_ncomp + t] = s;
                float mx = valid ? s : -INFINITY;
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                if (valid && (lane & (kBlk - 1)) == 0) block_max[(int64_t)b * ld_bm + t / kBlk] = mx;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acce[a]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && sh.abort) raise_status(dev_status, CSA2_DEV_TIMEOUT);
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    trace_end(kTraceIndex);
}

constexpr int kTcSmem = (int)sizeof(TcShared) + 1024;
static_assert(kTcSmem <= 227 * 1024, "shared memory of the tensor-core Indexer");

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

int check_index_args(const csa2_params* p, int B, int64_t max_ncomp, const void* q_vals,
                     const void* q_scales, const void* w, const void* key_cache,
                     const void* n_tokens, const void* scores, const void* block_max) {
    if (!p) return fail(CSA2_ERR_INVALID_ARG, "index_scores: params is NULL");
    if (B < 0 || max_ncomp < 0) return fail(CSA2_ERR_INVALID_ARG, "index_scores: negative size");
    if (p->index_heads != kHi || p->index_dim != kDi || p->block_size != kBlk ||
        p->compress_ratio < 1)
        return fail(CSA2_ERR_UNSUPPORTED, "index_scores: built for 32 heads x 128, blocks of 8");
    if (B == 0 || max_ncomp == 0) return -1;  // nothing to do
    if (!q_vals || !q_scales || !w || !key_cache || !n_tokens || !scores || !block_max)
        return fail(CSA2_ERR_INVALID_ARG, "index_scores: NULL buffer");
    if (!aligned16(q_vals) || !aligned16(w) || (reinterpret_cast<uintptr_t>(q_scales) & 7))
        return fail(CSA2_ERR_ALIGN, "index_scores: q_vals, w 16-byte, q_scales 8-byte aligned");
    return CSA2_OK;
}

}  // namespace

CSA2_TRACE_SETTER(trace_set_index)

cudaError_t preload_index() {
    cudaError_t e = preload_kernel(k_index_keys_write);
    if (!e) e = preload_kernel(k_index_scores_cc);
    if (!e) e = preload_kernel(k_index_scores_tc, kTcSmem);
    return e;
}

}  // namespace csa2

using namespace csa2;

extern "C" int csa2_index_keys_write(const csa2_params* p, int B, int64_t n, const uint8_t* vals,
                                     const uint8_t* scales, const int64_t* pos0,
                                     uint8_t* const* dst, const int64_t* cap, int32_t* dev_status,
                                     void* stream) {
    CSA2_CHECK_PARAMS(p);
    if (B < 0 || n < 0) return fail(CSA2_ERR_INVALID_ARG, "index_keys_write: negative size");
    if (p->index_dim != kDi) return fail(CSA2_ERR_UNSUPPORTED, "index_keys_write: built for Di=128");
    if (B == 0 || n == 0) return CSA2_OK;
    if (!vals || !scales || !pos0 || !dst || !cap)
        return fail(CSA2_ERR_INVALID_ARG, "index_keys_write: NULL buffer");
    if (!aligned16(vals) || (reinterpret_cast<uintptr_t>(scales) & 7))
        return fail(CSA2_ERR_ALIGN, "index_keys_write: vals 16-byte, scales 8-byte aligned");
    const int64_t total = (int64_t)B * n;
    if (const int rc = ensure_loaded()) return rc;
    k_index_keys_write<<<(unsigned)((total + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        B, n, vals, scales, pos0, dst, cap, dev_status);
    return check_launch("index_keys_write");
}

extern "C" int csa2_index_scores_cuda_cores(const csa2_params* p, int B, int64_t max_ncomp,
                                            const uint8_t* q_vals, const uint8_t* q_scales,
                                            const float* w, const uint8_t* const* key_cache,
                                            const int32_t* n_tokens, float* scores,
                                            float* block_max, int32_t* dev_status, void* stream) {
    const int rc = check_index_args(p, B, max_ncomp, q_vals, q_scales, w, key_cache, n_tokens,
                                    scores, block_max);
    if (rc != CSA2_OK) return rc < 0 ? CSA2_OK : rc;
    const int64_t gx = (max_ncomp + kKeysPerCta - 1) / kKeysPerCta;
    if (gx > 0x7fffffff) return fail(CSA2_ERR_UNSUPPORTED, "index_scores: too many positions");
    if (B > 65535) return fail(CSA2_ERR_UNSUPPORTED, "index_scores: at most 65535 sequences per call");
    if (const int rc = ensure_loaded()) return rc;
    k_index_scores_cc<<<dim3((unsigned)gx, B), kKeysPerCta, 0, static_cast<cudaStream_t>(stream)>>>(
        max_ncomp, p->compress_ratio, q_vals, q_scales, w, key_cache, n_tokens, scores, block_max,
        dev_status);
    return check_launch("index_scores_cuda_cores");
}

extern "C" int csa2_index_scores(const csa2_params* p, int B, int64_t max_ncomp,
                                 const uint8_t* q_vals, const uint8_t* q_scales, const float* w,
                                 const uint8_t* const* key_cache, const int32_t* n_tokens,
                                 float* scores, float* block_max, int32_t* dev_status,
                                 void* stream) {
    const int rc = check_index_args(p, B, max_ncomp, q_vals, q_scales, w, key_cache, n_tokens,
                                    scores, block_max);
    if (rc != CSA2_OK) return rc < 0 ? CSA2_OK : rc;
    if (B > 65535) return fail(CSA2_ERR_UNSUPPORTED, "index_scores: at most 65535 sequences per call");
    // loads the kernel and sets its shared-memory limit on this device, once per device
    if (const int rc = ensure_loaded()) return rc;
    const int64_t tiles_max = (int64_t)B * ((max_ncomp + kTilesPerStage * kKeyTile - 1) / (kTilesPerStage * kKeyTile));
    int64_t ctas = num_sms();
    if (p->max_ctas > 0 && p->max_ctas < ctas) ctas = p->max_ctas;
    const int grid = (int)std::min<int64_t>(tiles_max, ctas);
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kTcThreads);
        cfg.dynamicSmemBytes = kTcSmem;
        cfg.stream = static_cast<cudaStream_t>(stream);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, k_index_scores_tc, B, max_ncomp, p->compress_ratio, q_vals, q_scales, w,
                               key_cache, n_tokens, scores, block_max, dev_status) != cudaSuccess)
            return check_launch("index_scores");
    }
    return check_launch("index_scores");
}
