// Fused multi-layer sparse attention on the 5th-generation tensor cores
// (tcgen05): the decode query of each sequence attends to its 128-slot window
// and its 512 selected compressed positions, with a per-head sink logit in the
// denominator ("DeepSeek-V4.1-Flash-NVFP4" §3.4 gather + online softmax +
// attn_sink, §三 640 positions per query, §3.1 FP8 window, §一 one shared
// 512-d KV head so K = V = the latent, §四 reader layers share the source
// layer's compressed cache and selection).
//
// Work unit: one (layer, sequence); a persistent CTA per SM walks its units
// round robin, or (with a workspace) an equal contiguous range of (unit, tile)
// items, a unit cut by a range boundary being merged by log-sum-exp (see the
// schedule below). The 640 positions are 5 tiles of 128 (tiles 0..3 = idx[0..512) in 128s, tile
// 4 = the window ring: a unit opens on gathered rows, one round trip away, and
// the window's two rounds of loads overlap tile 3). Per tile, with the
// positions as the MMA's M:
//   S^T[128 x 64]  = K_tile[128 x 512] . Q^T            (TMEM, 64 columns)
//   O^T[512 x 64] += V_tile^T[512 x 128] . P^T[128 x 64] (TMEM, 4 x 64 columns)
// The tile is decoded exactly into f16 in shared memory once and is the A
// operand of both products: K-major for S (rows = positions), MN-major for PV
// (the latent dims run along the rows). E2M1 x E4M3 has at most 5 significant
// bits and E4M3 4, so both are exact in f16. The query is scaled per head by a
// power of two into f16 (exact except below 2^-24 of the head's largest
// element) and the factor is folded into the logit scale.
//
// Roles: 8 producer warps gather and decode rows (and stage Q), one thread
// issues every MMA, 8 softmax warps (4 TMEM lane quarters x 2 head halves)
// turn S into P in shared memory and finally read O out. The softmax keeps a
// per-head running maximum that only moves when a tile's maximum exceeds it by
// more than 2^8 (then the O columns of those heads are rescaled in TMEM), so P
// stays <= 256 and the common path never touches O. Every wait is bounded.
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace csa2 {
namespace {
using namespace sm100;

constexpr int kTiles = (kW + kKp) / 128;  // 5
constexpr int kSoftWarps = 8;
constexpr int kProdWarps = 8;
constexpr int kMmaWarp = kSoftWarps + kProdWarps;  // 16
constexpr int kAttnThreads = 32 * (kMmaWarp + 1);  // 544
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyMax = 8.0f;  // log2 of the largest P the lazy maximum allows

constexpr uint32_t kQChunk = 64 * 128;    // 64 heads x 64 dims (f16), one 128-byte row per head
constexpr uint32_t kKVChunk = 128 * 128;  // 128 positions x 64 dims
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O^T: 4 blocks of 128 dims x 64 heads
constexpr uint32_t kColS = 256;  // S^T: 128 positions x 64 heads

// Instruction descriptors (kind::f16): D fp32 (bits 4..5 = 1), A and B f16
// (bits 7..9, 10..12 = 0), N = 64 (N>>3 in bits 17..22), M = 128 (M>>4 in
// bits 24..28); bits 15 / 16 select MN-major A / B.
constexpr uint32_t kIdescS = (1u << 4) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescS | (1u << 15) | (1u << 16);

struct AttnShared {
    uint8_t q[8][kQChunk];    // B operand of S: Q[64 heads x 512] f16, 128-byte swizzle, K-major
    uint8_t kv[8][kKVChunk];  // the decoded tile [128 x 512] f16 in 8 column chunks, 128-byte swizzle
    uint8_t p[128 * 128];     // B operand of PV: P[128 positions x 64 heads] f16, MN-major
    float col_scale[2][64];   // per-head logit factor (softmax scale x log2 e / query scale), by unit parity
    float red_max[4][64];     // per lane quarter: the tile's maximum of each head
    float red_sum[4][64];     // per lane quarter: the sum over its 32 rows of each head
    // q_full[it & 1] publishes the query (and col_scale) of piece it. Two barriers:
    // a one-tile piece needs no softmax progress before its S completes, so the
    // producers can publish the next piece's query before the softmax warps have
    // waited on this one; on a single barrier two completed phases would read as
    // none. (Only a CTA's first piece can be that short and have a successor.)
    uint64_t q_full[2], q_empty, s_full, p_full, o_full, drain;
    uint64_t chunk_full[4], chunk_empty[4], red_max_bar[2], red_sum_bar[2];
    uint64_t soft_bar;  // the 8 softmax warps (merge of a cut unit)
    uint32_t tmem_base;
    int abort;
    int merge;          // merge decision of a cut unit, broadcast to the softmax warps
};
constexpr int kAttnSmem = (int)sizeof(AttnShared) + 1024;

// 16-byte unit u of row r in a 128-byte-swizzled region (8 units per row).
__device__ __forceinline__ uint32_t sw128(int r, int u) {
    return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t h2_lo(uint32_t h2) { return __byte_perm(h2, 0u, 0x1010); }
__device__ __forceinline__ uint32_t h2_hi(uint32_t h2) { return __byte_perm(h2, 0u, 0x3232); }

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Eight E2M1 codes (one word, element 0 in the low nibble) -> four f16 pairs, exact.
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t* o) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// Four E4M3 bytes (one word) -> two f16 pairs, exact.
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t* o) {
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
        " cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
        : "=r"(o[0]), "=r"(o[1])
        : "r"(w));
}

__device__ __forceinline__ uint32_t f32x2_to_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ bool win_row_valid(int r, int64_t T, int linear) {
    return T > 0 && (linear ? T - kW + r >= 0 : (T >= kW || (int64_t)r < T));
}

// Sum 16 per-head values over the 32 lanes of a warp; lane h returns head
// h mod 16. Each step hands half of the remaining heads to the partner lane,
// a last exchange adds the two lane halves (16 shuffles).
__device__ __forceinline__ float xreduce_sum16(float* v, int lane) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float keep = up ? v[i + o] : v[i];
            const float give = up ? v[i] : v[i + o];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;\n" : "=f"(r) : "f"(v));
    return r;
}

struct UnitArgs {
    int L, B, ratio, win_linear;
    int b0, nb;  // the sequences [b0, b0 + nb) of the batch of B are processed; units = L * nb
    int split;   // 0: whole units round robin; 1: even ranges of (unit, tile) items
    float* ws_part;   // split: per boundary two partial results (kPartFloats each)
    int32_t* ws_cnt;  // split: per boundary the count of its finished pieces
    float scale_log2;
    const __nv_bfloat16* q;
    const float* sink;
    const void* const* win;
    const int32_t* n_tokens;
    const void* const* comp;
    const uint8_t* const* comp_scales;
    const int32_t* idx;
    __nv_bfloat16* out;
    int32_t* dev_status;
};

// Unit u of a launch -> layer l, sequence b and the flat index l * B + b of the
// layer-major q / out / window arrays.
struct UnitIdx {
    int l, b, f;
};
__device__ __forceinline__ UnitIdx unit_idx(const UnitArgs& a, int u) {
    UnitIdx x;
    x.l = u / a.nb;
    x.b = a.b0 + u % a.nb;
    x.f = x.l * a.B + x.b;
    return x;
}

// ---------------------------------------------------------------- schedule
// A piece is the tiles [j0, j1) of unit u. Without a workspace a CTA takes whole
// units round robin (blockIdx.x, + gridDim.x, ...). With one, the L * nb * 5
// (unit, tile) items are cut into gridDim.x contiguous ranges of equal length,
// so every CTA streams the same number of tiles (10 or 11 of them for 320 units
// on 152 CTAs, against 3 or 2 whole units of 5). A unit cut by the start of
// CTA c's range is finished by two pieces — its head, the last piece of CTA
// c - 1, and its tail, the first piece of CTA c — which share boundary slot c.
// A range is at least 5 items long (grid <= units), so no unit is cut twice.
struct Piece {
    int u, j0, j1;
    // boundary slot of a cut unit (0: the unit is whole) and the piece's role
    // in it (0: head, tiles from 0; 1: tail, tiles up to 5)
    __device__ __forceinline__ int slot(const UnitArgs& a) const {
        if (!a.split) return 0;
        return j0 > 0 ? (int)blockIdx.x : (j1 < kTiles ? (int)blockIdx.x + 1 : 0);
    }
    __device__ __forceinline__ int role() const { return j0 > 0 ? 1 : 0; }
};

struct PieceIter {
    int item, end, step;  // step: items between round-robin units; 0 in range mode
    __device__ __forceinline__ void init(const UnitArgs& a) {
        const int64_t n = (int64_t)a.L * a.nb * kTiles;  // < 2^31 (units <= 2^28)
        if (a.split) {
            item = (int)(n * blockIdx.x / gridDim.x);
            end = (int)(n * (blockIdx.x + 1) / gridDim.x);
            step = 0;
        } else {
            item = (int)blockIdx.x * kTiles;
            end = (int)n;
            step = (int)gridDim.x * kTiles;
        }
    }
    __device__ __forceinline__ bool next(Piece& p) {
        if (item >= end) return false;
        p.u = item / kTiles;
        p.j0 = item - p.u * kTiles;
        p.j1 = min(kTiles, p.j0 + (end - item));
        item = step ? item + step : item + (p.j1 - p.j0);
        return true;
    }
};

// Partial result of a piece in its boundary slot: O [64 heads][512 dims] fp32
// (unnormalised, relative to the piece's running maximum), then the maximum m
// (log2 domain) and the sum l of each head.
constexpr int kPartFloats = kH * kD + 2 * kH;

__device__ __forceinline__ bool unit_aligned(const UnitArgs& a, int f, int b) {
    const uintptr_t w = reinterpret_cast<uintptr_t>(a.win[f]);
    const uintptr_t c = reinterpret_cast<uintptr_t>(a.comp[b]);
    const uintptr_t s = reinterpret_cast<uintptr_t>(a.comp_scales[b]);
    return ((w | c) & 15u) == 0 && (s & 3u) == 0;
}

// ---------------------------------------------------------------- producers
// Thread (r, hf) of the 256 producer threads owns row r of every tile and the
// column chunk 2*pair + hf of each pair of chunks (64 dims).
__device__ void producer_role(AttnShared& sh, const UnitArgs& a, int pt, int lane,
                              volatile int* abort) {
    const int pw = pt >> 5, r = pt >> 1, hf = pt & 1;
    PieceIter pi;
    pi.init(a);
    Piece pc;
    int it = 0, gt = 0;  // pieces and tiles done
    int64_t T = 0;
    bool aligned = false;
    int32_t xs[kTiles - 1];
    for (; pi.next(pc); ++it) {
        const UnitIdx ui = unit_idx(a, pc.u);
        const int b = ui.b;
        // ---- query: warp pw stages heads 8pw..8pw+7, lane = dims 16*lane..+15. The
        // loads go first: nothing below waits on them until the conversion, so their
        // latency overlaps the scalar loads and the wait for the last S of the
        // previous piece (no branch on a loaded value comes before that wait).
        {
            const uint4* qu = reinterpret_cast<const uint4*>(a.q + (int64_t)ui.f * kH * kD);
            uint4 qa[4], qb[4];
#pragma unroll
            for (int hi = 0; hi < 4; ++hi) {
                const uint4* src = qu + (int64_t)(8 * pw + hi) * (kD / 8) + 2 * lane;
                qa[hi] = __ldg(src);
                qb[hi] = __ldg(src + 1);
            }
            T = a.n_tokens[b];
            aligned = unit_aligned(a, ui.f, b);
            // selected positions of this thread's row in tiles 0..3
#pragma unroll
            for (int j = 0; j < kTiles - 1; ++j) xs[j] = a.idx[(int64_t)b * kKp + 128 * j + r];
            if (it > 0 && !mbar_wait(&sh.q_empty, (uint32_t)((it - 1) & 1), abort)) return;
            if (!aligned && pt == 0) raise_status(a.dev_status, CSA2_DEV_BAD_ALIGN);
#pragma unroll
            for (int hi = 0; hi < 8; ++hi) {
                const int h = 8 * pw + hi;
                const uint32_t w[8] = {qa[hi & 3].x, qa[hi & 3].y, qa[hi & 3].z, qa[hi & 3].w,
                                       qb[hi & 3].x, qb[hi & 3].y, qb[hi & 3].z, qb[hi & 3].w};
                if (hi < 4) {  // the second half of the heads: issue its loads now
                    const uint4* src = qu + (int64_t)(8 * pw + hi + 4) * (kD / 8) + 2 * lane;
                    qa[hi] = __ldg(src);
                    qb[hi] = __ldg(src + 1);
                }
                float f[16];
                float mx = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    f[2 * k] = __uint_as_float(w[k] << 16);
                    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
                    mx = fmaxf(mx, fmaxf(fabsf(f[2 * k]), fabsf(f[2 * k + 1])));
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                // 2^s with the head's largest |q| in [2^14, 2^15): f16 keeps 11 bits down to 2^-14
                int s = 14 - ((int)((__float_as_uint(mx) >> 23) & 0xffu) - 127);
                s = max(-126, min(126, s));
                const float two_s = __uint_as_float((uint32_t)(s + 127) << 23);
                uint32_t hq[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) hq[k] = f32x2_to_h2(f[2 * k] * two_s, f[2 * k + 1] * two_s);
                uint8_t* row = sh.q[lane >> 2];
                const int u0 = (lane & 3) * 2;
                *reinterpret_cast<uint4*>(row + sw128(h, u0)) = make_uint4(hq[0], hq[1], hq[2], hq[3]);
                *reinterpret_cast<uint4*>(row + sw128(h, u0 + 1)) = make_uint4(hq[4], hq[5], hq[6], hq[7]);
                if (lane == 0)
                    sh.col_scale[it & 1][h] = a.scale_log2 * __uint_as_float((uint32_t)(127 - s) << 23);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.q_full[it & 1]);

        // ---- the 5 tiles: the 4 tiles of selected rows, then the window
        const int64_t n_c = T > 0 ? T / a.ratio : 0;
        const uint8_t* winb = static_cast<const uint8_t*>(a.win[ui.f]);
        const uint8_t* compb = static_cast<const uint8_t*>(a.comp[b]);
        const uint8_t* compsb = a.comp_scales[b];
        for (int j = pc.j0; j < pc.j1; ++j, ++gt) {
            // window: two pairs in flight (4 x 16 B each); compressed: all four (2 x 16 B + scales)
            uint4 raw[8];
            uint32_t scw[4];
            bool valid;
            const uint4* wsrc = nullptr;
            if (j == kTiles - 1) {
                valid = aligned && win_row_valid(r, T, a.win_linear);
                wsrc = reinterpret_cast<const uint4*>(winb + (int64_t)r * kD + 64 * hf);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    raw[k] = valid ? __ldg(wsrc + 8 * (k >> 2) + (k & 3)) : make_uint4(0u, 0u, 0u, 0u);
            } else {
                const int64_t x0 = xs[j];
                if (x0 >= n_c && hf == 0) raise_status(a.dev_status, CSA2_DEV_BAD_INDEX);
                valid = aligned && x0 >= 0 && x0 < n_c;
                const int64_t x = valid ? x0 : 0;
                const uint4* src = reinterpret_cast<const uint4*>(compb + x * (kD / 2) + 32 * hf);
                const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(compsb + x * (kD / kGroup) + 4 * hf);
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {
                    raw[2 * pr] = valid ? __ldg(src + 4 * pr) : make_uint4(0u, 0u, 0u, 0u);
                    raw[2 * pr + 1] = valid ? __ldg(src + 4 * pr + 1) : make_uint4(0u, 0u, 0u, 0u);
                    scw[pr] = valid ? __ldg(ssrc + 2 * pr) : 0u;
                }
            }
#pragma unroll
            for (int pr = 0; pr < 4; ++pr) {
                if (gt > 0 && !mbar_wait(&sh.chunk_empty[pr], (uint32_t)((gt - 1) & 1), abort)) return;
                uint8_t* dst = sh.kv[2 * pr + hf];
                if (!valid) {
#pragma unroll
                    for (int un = 0; un < 8; ++un)
                        *reinterpret_cast<uint4*>(dst + sw128(r, un)) = make_uint4(0u, 0u, 0u, 0u);
                } else if (j == kTiles - 1) {  // 64 E4M3 bytes -> 64 f16, unit un = bytes 8un..8un+7
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 v = raw[4 * (pr & 1) + k];
                        uint32_t o[8];
                        e4m3x4_to_h2x2(v.x, &o[0]);
                        e4m3x4_to_h2x2(v.y, &o[2]);
                        e4m3x4_to_h2x2(v.z, &o[4]);
                        e4m3x4_to_h2x2(v.w, &o[6]);
                        *reinterpret_cast<uint4*>(dst + sw128(r, 2 * k)) = make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4*>(dst + sw128(r, 2 * k + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                    if (pr + 2 < 4) {  // refill the slot with pair pr + 2
#pragma unroll
                        for (int k = 0; k < 4; ++k) raw[4 * (pr & 1) + k] = __ldg(wsrc + 8 * (pr + 2) + k);
                    }
                } else {  // 32 E2M1 bytes (4 groups of 16) x E4M3 group scale -> 64 f16
                    const uint32_t w8[8] = {raw[2 * pr].x,     raw[2 * pr].y,     raw[2 * pr].z,
                                            raw[2 * pr].w,     raw[2 * pr + 1].x, raw[2 * pr + 1].y,
                                            raw[2 * pr + 1].z, raw[2 * pr + 1].w};
                    uint32_t s4[2];
                    e4m3x4_to_h2x2(scw[pr], s4);
                    const uint32_t sg[4] = {h2_lo(s4[0]), h2_hi(s4[0]), h2_lo(s4[1]), h2_hi(s4[1])};
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi) {  // word wi = 8 codes of group wi / 2 = unit wi
                        uint32_t o[4];
                        e2m1x8_to_h2x4(w8[wi], o);
                        *reinterpret_cast<uint4*>(dst + sw128(r, wi)) =
                            make_uint4(hmul2(o[0], sg[wi >> 1]), hmul2(o[1], sg[wi >> 1]),
                                       hmul2(o[2], sg[wi >> 1]), hmul2(o[3], sg[wi >> 1]));
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.chunk_full[pr]);
            }
        }
    }
}

// ---------------------------------------------------------------- MMA issuer
__device__ void mma_role(AttnShared& sh, const UnitArgs& a, uint32_t tmem, volatile int* abort) {
    // Descriptors are built once; a K step or a chunk moves only the start
    // address field (bits 0..13, address >> 4), which never carries out.
    const uint64_t dKV = smem_desc(smem_u32(sh.kv[0]), 16, 1024, kLayoutSw128);
    const uint64_t dQ = smem_desc(smem_u32(sh.q[0]), 16, 1024, kLayoutSw128);
    const uint64_t dV = smem_desc(smem_u32(sh.kv[0]), kKVChunk, 1024, kLayoutSw128);
    const uint64_t dP = smem_desc(smem_u32(sh.p), 1024, 1024, kLayoutSw128);
    PieceIter pi;
    pi.init(a);
    Piece pc;
    int it = 0, gt = 0;
    for (; pi.next(pc); ++it) {
        if (!mbar_wait(&sh.q_full[it & 1], (uint32_t)((it >> 1) & 1), abort)) return;
        tc_fence_after();
        for (int j = pc.j0; j < pc.j1; ++j, ++gt) {
            // S^T = K . Q^T over the 512 dims, chunk pair by chunk pair as they land
#pragma unroll
            for (int pr = 0; pr < 4; ++pr) {
                if (!mbar_wait(&sh.chunk_full[pr], (uint32_t)(gt & 1), abort)) return;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = 2 * pr + cc;
                        mma_f16(tmem + kColS, dKV + ((c * kKVChunk + 32 * k) >> 4),
                                dQ + ((c * kQChunk + 32 * k) >> 4), kIdescS, (pr | cc | k) != 0);
                    }
            }
            tc_commit(&sh.s_full);
            if (j == pc.j1 - 1) tc_commit(&sh.q_empty);
            // O^T += V^T . P^T, one block of 128 dims (= one chunk pair) at a time
            if (!mbar_wait(&sh.p_full, (uint32_t)(gt & 1), abort)) return;
            tc_fence_after();
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_f16(tmem + kColO + 64 * mb, dV + ((2 * mb * kKVChunk + k * 2048) >> 4),
                            dP + ((k * 2048) >> 4), kIdescPV, j != pc.j0 || k != 0);
                tc_commit(&sh.chunk_empty[mb]);
            }
        }
        tc_commit(&sh.o_full);
    }
}

// ---------------------------------------------------------------- softmax + epilogue
// Per-unit values a softmax thread needs, loaded one unit ahead.
struct SoftUnit {
    int32_t T, n_c;  // raw tokens, compressed positions
    bool aligned;
    float sink2;     // sink logit of head 32hh + lane, log2 domain
    int32_t xs[4];   // this row's selected positions in tiles 0..3
    __device__ __forceinline__ void load(const UnitArgs& a, int u, int r, int hh, int lane) {
        const UnitIdx ui = unit_idx(a, u);
        const int l = ui.l, b = ui.b;
        T = a.n_tokens[b];
        n_c = T > 0 ? T / a.ratio : 0;
        aligned = unit_aligned(a, ui.f, b);
        sink2 = a.sink[(int64_t)l * kH + 32 * hh + lane] * kLog2e;
#pragma unroll
        for (int j = 0; j < 4; ++j) xs[j] = a.idx[(int64_t)b * kKp + 128 * j + r];
    }
};

// Barrier of the 8 softmax warps on an mbarrier (bounded wait: an aborted warp
// cannot strand the others). n counts the phases used so far.
__device__ __forceinline__ bool soft_sync(AttnShared& sh, uint32_t& n, int lane, volatile int* abort) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.soft_bar);
    return mbar_wait(&sh.soft_bar, (n++) & 1u, abort);
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ void softmax_role(AttnShared& sh, const UnitArgs& a, uint32_t tmem, int warp, int lane,
                             volatile int* abort) {
    const int qd = warp & 3, hh = warp >> 2;
    const int r = 32 * qd + lane;                   // position row of the tile
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);  // this warp's TMEM lane quarter
    PieceIter pi;
    pi.init(a);
    Piece cur, nxt;
    bool has = pi.next(cur);
    bool has_nx = has && pi.next(nxt);
    SoftUnit cu, nx;
    if (has) cu.load(a, cur.u, r, hh, lane);
    int it = 0, gt = 0;
    uint32_t sync_n = 0;  // soft_sync phases used
    for (; has; ++it) {
        if (!mbar_wait(&sh.q_full[it & 1], (uint32_t)((it >> 1) & 1), abort)) return;
        float m_run = -INFINITY;  // running maximum of head 32hh + lane
        float lpart[32];          // this row's share of the sum of P, head 32hh + i
#pragma unroll
        for (int i = 0; i < 32; ++i) lpart[i] = 0.f;
        for (int j = cur.j0; j < cur.j1; ++j, ++gt) {
            const bool valid = j == kTiles - 1 ? cu.aligned && win_row_valid(r, cu.T, a.win_linear)
                                               : cu.aligned && cu.xs[j] >= 0 && cu.xs[j] < cu.n_c;
            if (j == cur.j1 - 1 && has_nx) nx.load(a, nxt.u, r, hh, lane);  // next piece's scalars, early
            if (!mbar_wait(&sh.s_full, (uint32_t)(gt & 1), abort)) return;
            tc_fence_after();
            const float bias = valid ? 0.f : -INFINITY;
            // this row's 32 logits (log2 domain), read from TMEM once per tile and kept
            // in registers for both passes
            float x[32];
            {
                uint32_t sv[32];
                tmem_ld_32x32b_x32(tl + kColS + 32 * hh, sv);
                const float4* cs = reinterpret_cast<const float4*>(&sh.col_scale[it & 1][32 * hh]);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 c = cs[q4];
                    x[4 * q4] = fmaf(__uint_as_float(sv[4 * q4]), c.x, bias);
                    x[4 * q4 + 1] = fmaf(__uint_as_float(sv[4 * q4 + 1]), c.y, bias);
                    x[4 * q4 + 2] = fmaf(__uint_as_float(sv[4 * q4 + 2]), c.z, bias);
                    x[4 * q4 + 3] = fmaf(__uint_as_float(sv[4 * q4 + 3]), c.w, bias);
                }
            }
            // warp maximum of every head (uniform in the warp); lane 0 publishes this
            // quarter's
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 m4 = make_float4(warp_max(x[4 * q4]), warp_max(x[4 * q4 + 1]),
                                              warp_max(x[4 * q4 + 2]), warp_max(x[4 * q4 + 3]));
                if (lane == 0) *reinterpret_cast<float4*>(&sh.red_max[qd][32 * hh + 4 * q4]) = m4;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.red_max_bar[hh]);
            if (!mbar_wait(&sh.red_max_bar[hh], (uint32_t)(gt & 1), abort)) return;
            const float tm = fmaxf(fmaxf(sh.red_max[0][32 * hh + lane], sh.red_max[1][32 * hh + lane]),
                                   fmaxf(sh.red_max[2][32 * hh + lane], sh.red_max[3][32 * hh + lane]));
            // lazy maximum: move only when this tile would push P above 2^kLazyMax
            const float m_new = tm > m_run + kLazyMax ? tm : m_run;
            const float alpha = (m_new != m_run && m_run != -INFINITY) ? ex2(m_run - m_new) : 1.f;
            const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
            m_run = m_new;
            const float mfix = m_run == -INFINITY ? 0.f : m_run;
            if (rescale) {
#pragma unroll
                for (int i = 0; i < 32; ++i) lpart[i] *= __shfl_sync(0xffffffffu, alpha, i);
            }
            // P = 2^(x - m), one 16-byte unit of the P row per 8 heads
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float pv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    pv[e] = ex2(x[8 * c8 + e] - __shfl_sync(0xffffffffu, mfix, 8 * c8 + e));
                    lpart[8 * c8 + e] += pv[e];
                }
                *reinterpret_cast<uint4*>(sh.p + sw128(r, 4 * hh + c8)) =
                    make_uint4(f32x2_to_h2(pv[0], pv[1]), f32x2_to_h2(pv[2], pv[3]),
                               f32x2_to_h2(pv[4], pv[5]), f32x2_to_h2(pv[6], pv[7]));
            }
            if (rescale) {  // O holds tiles < j (complete: S of tile j was issued after them)
#pragma unroll 1
                for (int blk = 0; blk < 4; ++blk) {
                    const uint32_t col = kColO + 64 * blk + 32 * hh;
                    uint32_t ov[32];
                    tmem_ld_32x32b_x32(tl + col, ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        ov[i] = __float_as_uint(__uint_as_float(ov[i]) * __shfl_sync(0xffffffffu, alpha, i));
                    tmem_st_32x32b_x32(tl + col, ov);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_full);
        }
        // ---- epilogue: o_h = O_h 2^{m-M} / (l 2^{m-M} + 2^{sink2-M}), M = max(m, sink2)
        if (!mbar_wait(&sh.o_full, (uint32_t)(it & 1), abort)) return;
        tc_fence_after();
        {
            const float lo = xreduce_sum16(lpart, lane), hi = xreduce_sum16(lpart + 16, lane);
            sh.red_sum[qd][32 * hh + lane] = lane < 16 ? lo : hi;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.red_sum_bar[hh]);
        if (!mbar_wait(&sh.red_sum_bar[hh], (uint32_t)(it & 1), abort)) return;
        const float lsum = (sh.red_sum[0][32 * hh + lane] + sh.red_sum[1][32 * hh + lane]) +
                           (sh.red_sum[2][32 * hh + lane] + sh.red_sum[3][32 * hh + lane]);
        const float sink2 = cu.sink2;
        // o = O fo (+ O' fx): fo scales this piece's O; fx the other piece's O' when a
        // unit cut at a CTA boundary is merged here (lane = head 32hh + lane).
        float fo = 0.f, fx = 0.f;
        const float* oth = nullptr;
        bool emit = true;
        const int slot = cur.slot(a);
        if (slot == 0) {
            const float M = fmaxf(m_run, sink2);
            const float sc = m_run == -INFINITY ? 0.f : exp2f(m_run - M);
            fo = sc / (lsum * sc + exp2f(sink2 - M));
        } else {
            // Cut unit: the piece that finishes second merges (log-sum-exp). A piece
            // that finds the other one counted already merges at once; otherwise it
            // publishes its partial (stores, fence, barrier, count) and the count
            // decides. The merging piece puts the count back to 0.
            float* slotp = a.ws_part + (int64_t)(slot - 1) * 2 * kPartFloats;
            float* own = slotp + cur.role() * kPartFloats;
            oth = slotp + (cur.role() ^ 1) * kPartFloats;
            int32_t* cnt = a.ws_cnt + (slot - 1);
            const bool t0 = warp == 0 && lane == 0;
            if (!soft_sync(sh, sync_n, lane, abort)) return;
            if (t0) sh.merge = ld_acquire_gpu(cnt) == 1 ? 1 : 0;
            if (!soft_sync(sh, sync_n, lane, abort)) return;
            int mode = sh.merge;
            if (mode == 0) {
                if (qd == 0) {
                    own[kH * kD + 32 * hh + lane] = m_run;
                    own[kH * kD + kH + 32 * hh + lane] = lsum;
                }
#pragma unroll 1
                for (int mb = 0; mb < 4; ++mb) {
                    uint32_t ov[32];
                    tmem_ld_32x32b_x32(tl + kColO + 64 * mb + 32 * hh, ov);
                    float* dst = own + (int64_t)(32 * hh) * kD + 128 * mb + 32 * qd + lane;
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[(int64_t)i * kD] = __uint_as_float(ov[i]);
                }
                __threadfence();
                if (!soft_sync(sh, sync_n, lane, abort)) return;
                if (t0) {
                    __threadfence();
                    sh.merge = atomicAdd(cnt, 1) == 1 ? 1 : 2;
                }
                if (!soft_sync(sh, sync_n, lane, abort)) return;
                mode = sh.merge;
            }
            emit = mode == 1;
            if (emit) {
                __threadfence();
                if (t0) *cnt = 0;
                const float mx = __ldcg(oth + kH * kD + 32 * hh + lane);
                const float lx = __ldcg(oth + kH * kD + kH + 32 * hh + lane);
                // combined head piece first whichever piece merges: the result does
                // not depend on which one finished second
                const bool own_head = cur.role() == 0;
                const float mh = own_head ? m_run : mx, lh = own_head ? lsum : lx;
                const float mt = own_head ? mx : m_run, lt = own_head ? lx : lsum;
                const float M = fmaxf(fmaxf(mh, mt), sink2);
                const float sh_ = mh == -INFINITY ? 0.f : exp2f(mh - M);
                const float st_ = mt == -INFINITY ? 0.f : exp2f(mt - M);
                const float den = __fadd_rn(__fadd_rn(__fmul_rn(lh, sh_), __fmul_rn(lt, st_)), exp2f(sink2 - M));
                fo = (own_head ? sh_ : st_) / den;
                fx = (own_head ? st_ : sh_) / den;
            }
        }
        // Lane = dim d = 128 mb + 32 qd + lane of 32 heads: for each head the warp
        // stores 32 consecutive bf16 (64 contiguous bytes) straight from registers.
        if (emit) {
            __nv_bfloat16* ob = a.out + (int64_t)unit_idx(a, cur.u).f * kH * kD + (int64_t)(32 * hh) * kD +
                                32 * qd + lane;
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
                uint32_t ov[32];
                tmem_ld_32x32b_x32(tl + kColO + 64 * mb + 32 * hh, ov);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    ov[i] = __float_as_uint(__fmul_rn(__uint_as_float(ov[i]), __shfl_sync(0xffffffffu, fo, i)));
                if (oth) {  // o = O_head f_head + O_tail f_tail, rounded products (no
                            // contraction), so the sum is the same whichever piece merges
                    const float* src = oth + (int64_t)(32 * hh) * kD + 128 * mb + 32 * qd + lane;
#pragma unroll
                    for (int h16 = 0; h16 < 2; ++h16) {
                        float x[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) x[i] = __ldcg(src + (int64_t)(16 * h16 + i) * kD);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            ov[16 * h16 + i] = __float_as_uint(__fadd_rn(
                                __uint_as_float(ov[16 * h16 + i]),
                                __fmul_rn(x[i], __shfl_sync(0xffffffffu, fx, 16 * h16 + i))));
                    }
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) ob[(int64_t)i * kD + 128 * mb] = __float2bfloat16_rn(__uint_as_float(ov[i]));
            }
        }
        cu = nx;
        cur = nxt;
        has = has_nx;
        has_nx = has && pi.next(nxt);
        tc_fence_before();
    }
}

__global__ void __launch_bounds__(kAttnThreads, 1) k_sparse_attn_tc(UnitArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // aligned by offsetting the shared array itself, so that accesses through sh
    // stay shared-space loads and stores
    AttnShared& sh = *reinterpret_cast<AttnShared*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &sh.abort;
    trace_start(kTraceAttn);
    if (tid == 0) {
        mbar_init(&sh.q_full[0], kProdWarps);
        mbar_init(&sh.q_full[1], kProdWarps);
        mbar_init(&sh.q_empty, 1);
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.p_full, kSoftWarps);
        mbar_init(&sh.o_full, 1);
        mbar_init(&sh.drain, 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&sh.chunk_full[i], kProdWarps);
            mbar_init(&sh.chunk_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.red_max_bar[i], 4);
            mbar_init(&sh.red_sum_bar[i], 4);
        }
        mbar_init(&sh.soft_bar, kSoftWarps);
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // Launched programmatically, the kernel before this one on the stream may still
    // be running: only the setup above (barriers, TMEM) overlaps it; every global
    // read comes after this wait.
    grid_dep_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp < kSoftWarps) {
        softmax_role(sh, a, tmem, warp, lane, abort);
    } else if (warp < kMmaWarp) {
        producer_role(sh, a, tid - 32 * kSoftWarps, lane, abort);
    } else if (lane == 0) {
        mma_role(sh, a, tmem, abort);
        // every MMA issued must finish before TMEM and shared memory are released
        tc_commit(&sh.drain);
        if (!mbar_wait_drain(&sh.drain, 0)) *abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && sh.abort) raise_status(a.dev_status, CSA2_DEV_TIMEOUT);
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    trace_end(kTraceAttn);
}

int sm_count(int dev) {
    static int n[64] = {0};
    if (dev < 0 || dev >= 64) return 1;
    if (!n[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        n[dev] = v > 0 ? v : 1;
    }
    return n[dev];
}

// Boundary slots a split launch of L x nb units uses on this device: one per CTA
// boundary of the grid the launch takes.
int64_t split_slots(const csa2_params* p, int64_t units, int dev) {
    int64_t sms = sm_count(dev);
    if (p->max_ctas > 0 && p->max_ctas < sms) sms = p->max_ctas;
    const int64_t grid = units < sms ? units : sms;
    return grid > 1 ? grid - 1 : 0;
}

size_t split_ws_bytes(int64_t slots) {
    const size_t cnt = ((size_t)slots * sizeof(int32_t) + 255) & ~(size_t)255;
    return cnt + (size_t)slots * 2 * kPartFloats * sizeof(float);
}

int launch_layers(const char* name, const csa2_params* p, int L, int B, int b0, int nb,
                  const void* q, const float* sink, const void* const* win,
                  const int32_t* n_tokens, const void* const* comp,
                  const uint8_t* const* comp_scales, const int32_t* idx, void* out,
                  void* workspace, size_t ws_bytes, bool split, int32_t* dev_status,
                  void* stream) {
    const std::string n(name);
    CSA2_CHECK_PARAMS(p);
    if (L < 0 || B < 0 || b0 < 0 || nb < 0 || b0 + nb > B)
        return fail(CSA2_ERR_INVALID_ARG, n + ": bad size or sequence range");
    if (L == 0 || nb == 0) return CSA2_OK;
    if (p->heads != kH || p->head_dim != kD || p->window != kW || p->topk_pos != kKp ||
        p->compress_ratio < 1)
        return fail(CSA2_ERR_UNSUPPORTED, n + ": built for 64 heads x 512, W=128, k=512");
    if (p->kv_format != CSA2_NVFP4 || p->win_format != CSA2_E4M3 || p->q_format != CSA2_BF16)
        return fail(CSA2_ERR_UNSUPPORTED, n + ": formats must be NVFP4, E4M3, BF16");
    if (!q || !sink || !win || !n_tokens || !comp || !comp_scales || !idx || !out)
        return fail(CSA2_ERR_INVALID_ARG, n + ": NULL buffer");
    if (!aligned16(q) || !aligned16(out))
        return fail(CSA2_ERR_ALIGN, n + ": q, out must be 16-byte aligned");
    if ((int64_t)L * B > (int64_t)1 << 28)
        return fail(CSA2_ERR_UNSUPPORTED, n + ": too many (layer, sequence) units");
    if (const int rc = ensure_loaded()) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return check_launch((n + ": device").c_str());
    const int64_t units = (int64_t)L * nb;
    if (split) {
        const int64_t slots = split_slots(p, units, dev);
        if (slots > 0 && !workspace) return fail(CSA2_ERR_INVALID_ARG, n + ": NULL workspace");
        if (ws_bytes < split_ws_bytes(slots))
            return fail(CSA2_ERR_INVALID_ARG, n + ": workspace smaller than its size function asks");
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(CSA2_ERR_ALIGN, n + ": workspace must be 256-byte aligned");
    }
    UnitArgs a;
    a.L = L;
    a.B = B;
    a.b0 = b0;
    a.nb = nb;
    a.ratio = p->compress_ratio;
    a.win_linear = p->win_layout == CSA2_WIN_LINEAR;
    a.scale_log2 = p->softmax_scale * kLog2e;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.sink = sink;
    a.win = win;
    a.n_tokens = n_tokens;
    a.comp = comp;
    a.comp_scales = comp_scales;
    a.idx = idx;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.dev_status = dev_status;
    a.split = split ? 1 : 0;
    a.ws_cnt = static_cast<int32_t*>(workspace);
    a.ws_part = nullptr;
    if (split && workspace) {
        const int64_t slots = split_slots(p, units, dev);
        a.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                             (split_ws_bytes(slots) - (size_t)slots * 2 * kPartFloats * sizeof(float)));
    }
    int64_t sms = sm_count(dev);
    if (p->max_ctas > 0 && p->max_ctas < sms) sms = p->max_ctas;
    const int grid = (int)(units < sms ? units : sms);
    // Programmatic launch: the CTAs may start while the kernel before it on the
    // stream still runs and do their setup (barriers, TMEM) on free SMs; the kernel
    // waits for that grid (grid_dep_wait) before any global read or write.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = kAttnSmem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_sparse_attn_tc, a) != cudaSuccess) return check_launch(name);
    return check_launch(name);
}

}  // namespace

CSA2_TRACE_SETTER(trace_set_attn_tc)

size_t sparse_attn_tc_ws_bytes(const csa2_params* p, int B) {
    int dev = 0;
    if (!p || B <= 0 || cudaGetDevice(&dev) != cudaSuccess) return 0;
    return split_ws_bytes(split_slots(p, B, dev));
}

int sparse_attn_tc_single(const char* name, const csa2_params* p, int B, const void* q,
                          const float* sink, const void* const* win, const int32_t* n_tokens,
                          const void* const* comp, const uint8_t* const* comp_scales,
                          const int32_t* idx, void* out, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return check_launch(name);
    const int64_t slots = split_slots(p, B, dev);
    if (ws_bytes < split_ws_bytes(slots) || (slots > 0 && !workspace))
        return fail(CSA2_ERR_SHAPE, std::string(name) + ": workspace smaller than the size query");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(CSA2_ERR_ALIGN, std::string(name) + ": workspace must be 256-byte aligned");
    if ((int64_t)B > (int64_t)1 << 28)
        return fail(CSA2_ERR_UNSUPPORTED, std::string(name) + ": too many sequences");
    if (const int rc = ensure_loaded()) return rc;
    // the completion counts of the cut units start at zero on every call, so the
    // caller's workspace needs no initialisation
    if (slots > 0 && cudaMemsetAsync(workspace, 0, (size_t)slots * sizeof(int32_t),
                                     static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return check_launch(name);
    return launch_layers(name, p, 1, B, 0, B, q, sink, win, n_tokens, comp, comp_scales, idx, out,
                         workspace, ws_bytes, true, dev_status, stream);
}

cudaError_t preload_attn_tc() { return preload_kernel(k_sparse_attn_tc, kAttnSmem); }

}  // namespace csa2

using namespace csa2;

extern "C" int csa2_sparse_attn_layers_part(const csa2_params* p, int L, int B, int b0, int nb,
                                            const void* q, const float* sink, const void* const* win,
                                            const int32_t* n_tokens, const void* const* comp,
                                            const uint8_t* const* comp_scales, const int32_t* idx,
                                            void* out, int32_t* dev_status, void* stream) {
    return launch_layers("sparse_attn_layers", p, L, B, b0, nb, q, sink, win, n_tokens, comp,
                         comp_scales, idx, out, nullptr, 0, false, dev_status, stream);
}

extern "C" int csa2_sparse_attn_layers(const csa2_params* p, int L, int B, const void* q,
                                       const float* sink, const void* const* win,
                                       const int32_t* n_tokens, const void* const* comp,
                                       const uint8_t* const* comp_scales, const int32_t* idx,
                                       void* out, int32_t* dev_status, void* stream) {
    return launch_layers("sparse_attn_layers", p, L, B, 0, B, q, sink, win, n_tokens, comp,
                         comp_scales, idx, out, nullptr, 0, false, dev_status, stream);
}

extern "C" size_t csa2_sparse_attn_layers_split_workspace_size(const csa2_params* p, int L, int B) {
    if (!p || L <= 0 || B <= 0) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return split_ws_bytes(split_slots(p, (int64_t)L * B, dev));
}

extern "C" int csa2_sparse_attn_layers_split(const csa2_params* p, int L, int B, const void* q,
                                             const float* sink, const void* const* win,
                                             const int32_t* n_tokens, const void* const* comp,
                                             const uint8_t* const* comp_scales, const int32_t* idx,
                                             void* out, void* workspace, size_t ws_bytes,
                                             int32_t* dev_status, void* stream) {
    return launch_layers("sparse_attn_layers_split", p, L, B, 0, B, q, sink, win, n_tokens, comp,
                         comp_scales, idx, out, workspace, ws_bytes, true, dev_status, stream);
}
