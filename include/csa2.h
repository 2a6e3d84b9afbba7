/*
 * csa2.h — C ABI of the CSA2 (Compressed Sparse Attention 2) hot path on GB300.
 *
 * One layer's decode path, as the "DeepSeek-V4.1-Flash-NVFP4" walkthrough
 * (lpnh.cn) describes it:
 *   csa2_compress_append   §3.2 Compressor (2:1 softmax-gated pooling, NVFP4
 *                          cache, pending half-pair kept in state) and §3.1
 *                          128-slot FP8 ring window, one write per token;
 *   csa2_index_scores      §3.3 Indexer (32 FP4 index heads, ReLU, per-head
 *                          weights) with the block maximum over 8 positions;
 *   csa2_select_topk       §3.3 select_candidate_blocks (top-2048 blocks of 8,
 *                          newest block kept) then top-512 positions;
 *   csa2_sparse_attn       §3.4 sparse_attn (gather, online softmax, attn_sink),
 *                          §三 128 window + 512 selected = 640 positions.
 * Sizes from the "CSA2稀疏注意力、384专家MoE与1M上下文" config walkthrough
 * (nxmr.cn) §2.1 and §一 (64 query heads sharing one KV head of dim 512).
 *
 * Conventions (all calls):
 *  - Pointers named *_dev (and every array argument unless stated otherwise)
 *    are CUDA device pointers. The caller owns every buffer; the library
 *    allocates nothing and keeps no per-call state. Scratch, where a call
 *    needs it, is a caller buffer sized by a *_workspace_size query.
 *  - Per-sequence caches are reached through device arrays of per-sequence
 *    base pointers (ragged batches need no common stride).
 *  - `stream` is a cudaStream_t passed as void*. Every call only enqueues work
 *    on it and returns; nothing synchronises. Stream order holds as usual: some
 *    kernels (the appends, the tensor-core Indexer, the fused attention) are
 *    programmatic launches whose blocks may be placed while the kernel ahead on
 *    the stream still runs, but they read and write nothing before it has
 *    completed.
 *  - Return value: CSA2_OK or a CSA2_ERR_* code for errors found on the host
 *    (bad arguments, unsupported sizes, launch failures; text in
 *    csa2_last_error(), per calling thread). Nothing is enqueued on error.
 *  - Errors only visible on the device (an index outside the cache, a length
 *    beyond capacity) set CSA2_DEV_* bits in the caller's int32 `dev_status`
 *    (atomicOr; may be NULL to skip), the offending element is skipped, and
 *    the kernel completes. The caller reads it after synchronising.
 *  - The hot kernels are specialised for the pages' sizes (csa2_default_params);
 *    other sizes return CSA2_ERR_UNSUPPORTED.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define CSA2_OK 0
#define CSA2_ERR_INVALID_ARG 1 /* NULL where a buffer is required, negative size */
#define CSA2_ERR_SHAPE 2       /* inconsistent sizes (e.g. workspace too small) */
#define CSA2_ERR_ALIGN 3       /* pointer not 16-byte aligned where vector loads need it */
#define CSA2_ERR_UNSUPPORTED 4 /* sizes or formats the kernels are not built for */
#define CSA2_ERR_CUDA 5        /* a CUDA launch or attribute call failed */

/* ---- device status bits (OR-ed into *dev_status) ---- */
#define CSA2_DEV_BAD_INDEX 1   /* a selected index >= the sequence's compressed length */
#define CSA2_DEV_BAD_LENGTH 2  /* a sequence length beyond the stated capacity, or < 0 */
#define CSA2_DEV_TIMEOUT 4     /* a pipeline wait gave up (the kernel returned early) */
#define CSA2_DEV_BAD_ALIGN 8   /* a per-sequence buffer base is misaligned (its rows read as empty) */

/* ---- formats ---- */
#define CSA2_F32 0   /* fp32 */
#define CSA2_NVFP4 1 /* E2M1 pairs (element 2k = low nibble of byte k) + one E4M3 scale per 16 */
#define CSA2_E4M3 2  /* FP8 E4M3 ("fn": max 448, no inf), unit scale */
#define CSA2_BF16 3  /* bfloat16 */

typedef struct csa2_params {
    int heads;            /* query heads sharing the KV head: 64 */
    int head_dim;         /* KV latent / query head dim D: 512 */
    int index_heads;      /* Indexer query heads: 32 */
    int index_dim;        /* Indexer head dim: 128 */
    int window;           /* ring window slots W: 128 */
    int block_size;       /* positions per candidate block: 8 */
    int topk_blocks;      /* blocks kept: 2048 */
    int topk_pos;         /* positions kept: 512 */
    int compress_ratio;   /* raw tokens per compressed position: 2 (the pooled 2:1
                             layers) or 1 (the 1:1 layers: pooling skipped, raw token
                             p is compressed row p) */
    int kv_format;        /* compressed cache: CSA2_NVFP4 (or CSA2_F32, unquantised) */
    int win_format;       /* window ring: CSA2_E4M3 (or CSA2_F32) */
    int q_format;         /* query and output: CSA2_BF16 (or CSA2_F32) */
    float softmax_scale;  /* logit scale: 1/sqrt(head_dim) */
    int win_layout;       /* window rows: CSA2_WIN_RING (row r = ring slot r, the
                             newest raw position p < T with p mod W = r) or
                             CSA2_WIN_LINEAR (row r = raw position T-W+r; used by
                             prefill, where each query has its own window) */
    int max_ctas;         /* upper bound on the CTAs of the persistent kernels
                             (csa2_index_scores, csa2_sparse_attn_layers); 0 = one
                             per SM. A caller that runs two of them concurrently on
                             different streams splits the SMs with it. Also
                             csa2_select_topk spreads each sequence over a cluster
                             of 4 CTAs only when 4 B <= max_ctas (0: 2 x SMs). */
    /* Rotary embedding of the compressed KV, applied by csa2_compress_append
     * ("CSA2稀疏注意力、384专家MoE与1M上下文" §2.2 compress_rope_theta, §四
     * rope_scaling yarn; "DeepSeek-V4.1-Flash-NVFP4" §3.2). Compressed row j is
     * rotated at raw position compress_ratio*j (its first raw token) after
     * pooling and before quantising: its last rope_dim dims, in adjacent pairs
     * (2i, 2i+1) -> (a cos - b sin, a sin + b cos) with angle pos*theta_i, where
     * theta_i is the YaRN "NTK-by-parts" frequency (Peng et al. 2023) of the
     * RoFormer frequency rope_theta^(-2i/rope_dim): with r_i = rope_orig_len *
     * theta_i / (2 pi) rotations over the original context, pairs with r_i >
     * rope_beta_fast keep theta_i, pairs with r_i < rope_beta_slow take
     * theta_i / rope_factor, and in between the two blend linearly in r_i.
     * Angles, sines and cosines in fp64; the rotated values are rounded to fp32.
     * The window is not rotated here (its tokens arrive rotated). */
    int rope_dim;         /* rotated dims: 0 (default: rows arrive rotated) or a
                             multiple of 4 up to head_dim */
    float rope_theta;     /* rotary base: 160000 */
    float rope_factor;    /* YaRN factor: 16 (1 = plain RoPE) */
    float rope_orig_len;  /* YaRN original context length: 65536 */
    float rope_beta_fast; /* 32 */
    float rope_beta_slow; /* 1 */
} csa2_params;

#define CSA2_WIN_RING 0
#define CSA2_WIN_LINEAR 1

/* Fills *p with the pages' configuration (64/512/32/128/128/8/2048/512/2,
 * NVFP4 cache, E4M3 window, bf16 query, 1/sqrt(512), ring window; rotary base
 * 160000, YaRN factor 16 over 65536 with betas 32/1, rope_dim 0 = rows arrive
 * rotated). */
void csa2_default_params(csa2_params* p);

/*
 * csa2_trace_attach — launch trace for diagnosing device errors. (No counterpart
 * in the pages.) record: NULL (off, the default) or a device-accessible pointer
 * to 4 int32, normally pinned host memory (with unified addressing the host
 * pointer is the device pointer), zero-filled by the caller. While attached,
 * one thread of each compress_append, index_scores (tcgen05), select_topk and
 * sparse_attn_layers* launch stores {kernel id, launch number} into words 0-1 when
 * the launch starts and into words 2-3 when its first CTA finishes (ids: 1
 * compress, 2 index, 3 select, 4 attention; launch numbers count per kernel).
 * After an error has ended the CUDA context the host can still read the record:
 * words 0-1 name the last launch that started. Applies to the current device;
 * returns CSA2_OK or CSA2_ERR_CUDA.
 */
int csa2_trace_attach(int32_t* record);

/* Library ABI version (major*10000 + minor*100 + patch). */
int csa2_version(void);

/* Text of the last host-side error on the calling thread ("" if none). */
const char* csa2_last_error(void);

/*
 * csa2_compress_append — append n_new raw tokens to B sequences of one layer.
 * ("DeepSeek-V4.1-Flash-NVFP4" §3.2 Compressor, §3.1 window.)
 *
 * Before the call sequence b holds T_b = n_tokens[b] raw tokens; compressed
 * row j pools raw tokens 2j and 2j+1; when T_b is odd, token T_b-1 waits in
 * pend_kv/pend_gate. For every pair completed by the new tokens, per channel d:
 *   alpha_i = softmax_{i in pair}(gate[i,d]),  c[d] = sum_i alpha_i * kv[i,d]  (fp32)
 * and c is written to compressed row j of comp[b]:
 *   kv_format NVFP4: per 16-channel group, S = E4M3(amax/6) (fp32 division,
 *     round to nearest even, saturating), codes = E2M1(c/S) (IEEE fp32
 *     division, RNE, saturating to +-6, sign kept), all codes 0 when S = 0.
 *     Row layout: comp[b] + j*D/2 bytes (values), comp_scales[b] + j*D/16 bytes.
 *   kv_format F32: comp[b] + j*D floats.
 * Every new raw token p also writes ring slot p mod W of win[b] (D bytes E4M3,
 * RNE satfinite, or D floats) — only the newest W of them, as the ring keeps.
 * Afterwards n_tokens[b] = T_b + n_new.
 * With compress_ratio 1 (the 1:1 layers, "CSA2稀疏注意力、384专家MoE与1M上下文"
 * §2.2) pooling is skipped: new raw token p is written as compressed row p with
 * the same encoding, and gate_new / pend_kv / pend_gate are not used.
 * With rope_dim > 0 each compressed row is rotated before it is encoded (see
 * csa2_params); rope_dim must be a multiple of 4 up to D and the YaRN settings
 * must have rope_theta > 0, rope_factor > 0, rope_orig_len > 0 and
 * rope_beta_fast > rope_beta_slow (else CSA2_ERR_UNSUPPORTED / INVALID_ARG).
 *
 *   kv_new, gate_new  [B, n_new, D] fp32, device. gate_new may be NULL when
 *                     comp is NULL or compress_ratio is 1.
 *   pend_kv, pend_gate [B, D] fp32, device; caller zero-initialises once
 *                     (may be NULL at compress_ratio 1).
 *   comp              device array [B] of per-sequence row bases, or NULL for a
 *                     window-only layer (compress ratio 0, or a layer that reads
 *                     another layer's compressed cache).
 *   comp_scales       device array [B] of scale-row bases (NVFP4 only).
 *   comp_cap          [B] int64, device: rows allocated per sequence; a row
 *                     j >= comp_cap[b] is not written and sets CSA2_DEV_BAD_LENGTH.
 *   win               device array [B] of ring bases ([W, D]).
 *   n_tokens          [B] int32, device, read and advanced.
 * Constraints: D == 512; compress_ratio 2 or 1; n_new >= 0; 16-byte aligned rows.
 */
int csa2_compress_append(const csa2_params* p, int B, int n_new,
                         const float* kv_new, const float* gate_new,
                         float* pend_kv, float* pend_gate,
                         void* const* comp, uint8_t* const* comp_scales, const int64_t* comp_cap,
                         void* const* win, int32_t* n_tokens,
                         int32_t* dev_status, void* stream);

/*
 * csa2_window_linear — the FP8 window rows a prefill chunk's queries attend to,
 * laid out linearly ("DeepSeek-V4.1-Flash-NVFP4" §3.1: the window holds the
 * newest 128 raw tokens, FP8). Call it before csa2_compress_append appends the
 * chunk. For each sequence b with T = n_tokens[b] tokens so far, writes
 * out[b] rows i = 0 .. W-1+n_new-1 with row i = raw position T-(W-1)+i:
 * the last W-1 positions before the chunk copied from the ring win[b] (rows of
 * positions < 0 are zero) followed by the n_new chunk tokens cast to E4M3 (RNE,
 * saturating). The query at raw position p then finds its window (positions
 * p-W+1..p) at row p-T of out[b], in the CSA2_WIN_LINEAR layout.
 *   kv_new [B, n_new, D] fp32; win: device array [B] of rings; n_tokens [B];
 *   out [B, W-1+n_new, D] bytes (E4M3 windows only).
 */
int csa2_window_linear(const csa2_params* p, int B, int n_new, const float* kv_new,
                       const void* const* win, const int32_t* n_tokens, uint8_t* out,
                       void* stream);

/*
 * csa2_nvfp4_quantize — quantise n_rows rows of row_len fp32 values to NVFP4
 * with exactly the rule csa2_compress_append uses ("DeepSeek-V4.1-Flash-NVFP4"
 * §3.2). Used for index keys/queries produced outside the path and to check
 * the quantiser on identical inputs.
 *   x      [n_rows, row_len] fp32, device;  vals [n_rows, row_len/2] bytes;
 *   scales [n_rows, row_len/16] bytes.  row_len % 16 == 0.
 */
int csa2_nvfp4_quantize(const float* x, int64_t n_rows, int row_len,
                        uint8_t* vals, uint8_t* scales, void* stream);

/*
 * Index-key cache layout (one per sequence). Positions are grouped in tiles of
 * 128; tile j (positions 128j..128j+127) is CSA2_KEY_TILE_BYTES = 9216
 * contiguous bytes, the exact shared-memory image the tensor-core Indexer
 * consumes, so one bulk copy moves a tile:
 *   bytes [0, 8192): E2M1 codes, 64 bytes per position m = t mod 128 (dim 2k in
 *     the low nibble of byte k), K-major with the 64-byte swizzle: byte b of
 *     16-byte chunk c of position m sits at  m*64 + ((c ^ ((m >> 1) & 3)) << 4) + b;
 *   bytes [8192, 9216): E4M3 group scales, group g (dims 16g..16g+15) of
 *     position m at  8192 + (g >> 2)*512 + (m & 31)*16 + (m >> 5)*4 + (g & 3).
 * A sequence holding n positions needs ceil(n/128) tiles. Rows past n in the
 * last tile are ignored. csa2_index_keys_write fills it from plain rows.
 */
#define CSA2_KEY_TILE 128
#define CSA2_KEY_TILE_BYTES 9216

/*
 * csa2_index_keys_write — write n plain NVFP4 index keys per sequence into the
 * tiled index-key caches (layout above), at positions pos0[b] .. pos0[b]+n-1.
 * ("DeepSeek-V4.1-Flash-NVFP4" §3.3: the shared FP4 index key the index heads
 * score; the keys come from a projection outside this path.)
 *   vals   [B, n, Di/2] bytes, scales [B, n, Di/16] bytes (plain NVFP4 rows, as
 *          csa2_nvfp4_quantize produces them), device;
 *   pos0   [B] int64, device;  dst: device array [B] of tiled cache bases;
 *   cap    [B] int64, device: positions each cache holds (tiles*128); a
 *          position >= cap[b] is skipped and sets CSA2_DEV_BAD_LENGTH.
 * Constraints: Di == 128.
 */
int csa2_index_keys_write(const csa2_params* p, int B, int64_t n,
                          const uint8_t* vals, const uint8_t* scales, const int64_t* pos0,
                          uint8_t* const* dst, const int64_t* cap,
                          int32_t* dev_status, void* stream);

/*
 * csa2_index_scores — decode Indexer over every compressed position of B
 * sequences ("DeepSeek-V4.1-Flash-NVFP4" §3.3):
 *   s_t = sum_{h<Hi} w[h] * ReLU( sum_{d<Di} q[h,d] * k[t,d] ),  t < n_c,
 * with q and k the NVFP4-decoded values (E2M1 code x E4M3 group scale), fp32
 * accumulation, and the block maximum m_b = max_{t in [8b, 8b+8), t < n_c} s_t.
 * n_c = n_tokens[b] / compress_ratio, clipped to max_ncomp.
 * Runs on the 5th-generation tensor cores (block-scaled FP4 MMA, 128 positions
 * x 32 heads per instruction pair), one CTA per SM streaming tiles.
 *
 *   q_vals   [B, Hi, Di/2] bytes   q_scales [B, Hi, Di/16] bytes   w [B, Hi] fp32
 *   key_cache device array [B] of tiled index-key caches (layout above); the
 *            cache of sequence b must hold ceil(n_c/128) tiles.
 *   scores   [B, max_ncomp] fp32 out (entries >= n_c untouched)
 *   block_max [B, ceil(max_ncomp/8)] fp32 out (entries >= ceil(n_c/8) untouched)
 *   max_ncomp >= every n_c (else CSA2_DEV_BAD_LENGTH, and the sequence is clipped).
 *   A pipeline wait that does not complete within about a second sets
 *   CSA2_DEV_TIMEOUT and the kernel returns.
 * Constraints: Hi == 32, Di == 128, block_size == 8, B <= 65535.
 * The fp32 result is exact (independent of summation order) when every
 * partial sum is a multiple of a common power of two below 2^24 of it — true
 * for E2M1 codes with power-of-two scales and weights.
 */
int csa2_index_scores(const csa2_params* p, int B, int64_t max_ncomp,
                      const uint8_t* q_vals, const uint8_t* q_scales, const float* w,
                      const uint8_t* const* key_cache,
                      const int32_t* n_tokens, float* scores, float* block_max,
                      int32_t* dev_status, void* stream);

/*
 * csa2_index_scores_shared — the Indexer for Q queries that all score ONE key
 * stream (the prefill chunk: every query of the chunk reads the same
 * sequence's index keys, up to its own causal length). Same per-query
 * contract as csa2_index_scores ("DeepSeek-V4.1-Flash-NVFP4" §3.3): for query
 * i, n_c(i) = n_tokens[i] / compress_ratio (clipped to max_ncomp with
 * CSA2_DEV_BAD_LENGTH), s_t = sum_h w[i,h] * ReLU(q_i,h . k_t) for t < n_c(i),
 * scores [Q, max_ncomp] fp32 and block_max [Q, ceil(max_ncomp/8)] fp32 written
 * for t < n_c(i) and its blocks. Because the keys are shared, scoring is a
 * dense block-scaled FP4 GEMM on the tensor cores: each 128-position key tile is
 * loaded once per 16 queries and multiplied with 4 queries x 32 heads per MMA.
 *   q_vals [Q, 32, 64] u8, q_scales [Q, 32, 8] u8 (E4M3), w [Q, 32] fp32
 *   key_cache  ONE tiled key cache (the layout of csa2_index_keys_write), device,
 *              16-byte aligned, with at least ceil(max n_c / 128) tiles.
 *   n_tokens   [Q] int32, device: raw context length seen by each query.
 * Work spans ceil(Q / 16) query blocks x ceil(max_ncomp / 512) key super-tiles;
 * the super-tiles past a block's longest query are skipped.
 */
int csa2_index_scores_shared(const csa2_params* p, int Q, int64_t max_ncomp,
                             const uint8_t* q_vals, const uint8_t* q_scales, const float* w,
                             const uint8_t* key_cache, const int32_t* n_tokens,
                             float* scores, float* block_max, int32_t* dev_status, void* stream);

/*
 * csa2_index_scores_cuda_cores — the same Indexer on CUDA cores (fp32 FMA, one
 * thread per position). Same arguments and results; kept to validate the
 * tensor-core build and as its ablation.
 */
int csa2_index_scores_cuda_cores(const csa2_params* p, int B, int64_t max_ncomp,
                                 const uint8_t* q_vals, const uint8_t* q_scales, const float* w,
                                 const uint8_t* const* key_cache,
                                 const int32_t* n_tokens, float* scores, float* block_max,
                                 int32_t* dev_status, void* stream);

/*
 * csa2_select_topk — two-level selection ("DeepSeek-V4.1-Flash-NVFP4" §3.3).
 * Per sequence, with n_c = n_tokens[b]/compress_ratio and n_b = ceil(n_c/8):
 *   if n_b > topk_blocks: keep block n_b-1 (it holds the newest position) and
 *   the best topk_blocks-1 other blocks by (block_max desc, block asc); else
 *   keep every block. Among the positions of kept blocks keep the best
 *   topk_pos by (score desc, position asc).
 *   idx   [B, topk_pos] int32 out: kept positions ascending, then -1 padding.
 *   n_sel [B] int32 out: number of valid entries (may be NULL).
 * Scores compare as fp32 values (-0 == +0). Ties are resolved exactly.
 * Because the block score is its best position's and topk_blocks - 1 >=
 * topk_pos, the result is the topk_pos best positions of the sequence; the
 * kernel finds them among the positions of the blocks whose maximum reaches a
 * sampled threshold that at least topk_pos block maxima reach. A small batch
 * (4 B <= max_ctas, or 2 x SMs) runs each sequence on a cluster of 4 CTAs that
 * share the pass over the block maxima through distributed shared memory; a
 * batch of more sequences than SMs runs a 512-thread build, two CTAs per SM.
 */
int csa2_select_topk(const csa2_params* p, int B, int64_t max_ncomp,
                     const float* scores, const float* block_max, const int32_t* n_tokens,
                     int32_t* idx, int32_t* n_sel, int32_t* dev_status, void* stream);

/* Bytes of scratch csa2_sparse_attn needs for a batch of B queries. */
size_t csa2_sparse_attn_workspace_size(const csa2_params* p, int B);

/*
 * csa2_sparse_attn — attention of one decode query per sequence over its
 * window and its selected compressed positions, with a per-head sink logit in
 * the denominator ("DeepSeek-V4.1-Flash-NVFP4" §3.4, §三, §3.1):
 *   attended set: raw positions max(0,T-W)..T-1 (ring slot p mod W of win[b],
 *   T = n_tokens[b]) and compressed rows idx[b][k] >= 0 of comp[b];
 *   z_j = softmax_scale * q_h . k_j;  o_h = sum_j e^{z_j} v_j / (e^{sink_h} + sum_j e^{z_j}),
 *   with K = V = the stored latent (NVFP4/E4M3 decoded exactly).
 *   q    [B, H, D] bf16 (or fp32)      sink [H] fp32     out [B, H, D] bf16 (or fp32)
 *   idx  [B, topk_pos] int32 (-1 = empty); an idx >= T/compress_ratio is
 *        skipped and sets CSA2_DEV_BAD_INDEX.
 *   workspace: device scratch of at least csa2_sparse_attn_workspace_size(p, B)
 *   bytes, 256-byte aligned (partial results of the schedule below); contents
 *   need no initialisation (the call clears what must start at zero, on the
 *   stream). Calls that share a workspace must be ordered (one stream or events).
 * Quantised formats (NVFP4 cache, E4M3 window, bf16 q/out) run on the tcgen05
 * tensor cores: the kernel of csa2_sparse_attn_layers_split with one layer
 * (f16 operands decoded exactly, fp32 accumulation in TMEM). The fp32 formats
 * run on CUDA cores in 5 position splits per sequence merged by log-sum-exp.
 * Constraints: H == 64, D == 512, W == 128, topk_pos == 512.
 */
int csa2_sparse_attn(const csa2_params* p, int B,
                     const void* q, const float* sink,
                     const void* const* win, const int32_t* n_tokens,
                     const void* const* comp, const uint8_t* const* comp_scales,
                     const int32_t* idx, void* out,
                     void* workspace, size_t ws_bytes,
                     int32_t* dev_status, void* stream);

/*
 * csa2_sparse_attn_mma — csa2_sparse_attn on the legacy warp-level tensor-core
 * path for the quantised formats (mma.sync bf16: 5 position splits per sequence
 * with partials in the workspace, then a log-sum-exp merge; P rounded to bf16).
 * Same arguments, workspace and results; kept as a second, independent
 * implementation and ablation of the tcgen05 path. fp32 formats as csa2_sparse_attn.
 */
int csa2_sparse_attn_mma(const csa2_params* p, int B,
                         const void* q, const float* sink,
                         const void* const* win, const int32_t* n_tokens,
                         const void* const* comp, const uint8_t* const* comp_scales,
                         const int32_t* idx, void* out,
                         void* workspace, size_t ws_bytes,
                         int32_t* dev_status, void* stream);

/*
 * csa2_sparse_attn_layers — csa2_sparse_attn for L layers that share one
 * compressed cache and one selection ("DeepSeek-V4.1-Flash-NVFP4" §四: the
 * KV-source layers' compressed cache is read by the layers in between; §3.3:
 * a published top-k is reused), each with its own query, window and sink.
 * Same arithmetic as csa2_sparse_attn, on the tcgen05 tensor cores: a
 * persistent CTA per SM takes (layer, sequence) units and streams their 640
 * positions with an online softmax, so it needs no workspace. Decoded rows
 * and P are 16-bit (f16) MMA operands with fp32 accumulation; the query is
 * scaled per head by a power of two into f16.
 *   q    [L, B, H, D] bf16      sink [L, H] fp32      out [L, B, H, D] bf16
 *   win  device array [L*B] of ring bases, layer-major (entry l*B + b)
 *   n_tokens [B]: raw tokens of sequence b (the same in every layer: the layers
 *        process one token stream); comp, comp_scales [B]; idx [B, topk_pos].
 *   Bases win[l*B+b] and comp[b] must be 16-byte aligned and comp_scales[b]
 *   4-byte aligned; a misaligned base sets CSA2_DEV_BAD_ALIGN and that unit's
 *   rows read as empty. q and out 16-byte aligned (else CSA2_ERR_ALIGN).
 * Constraints: H == 64, D == 512, W == 128, topk_pos == 512, NVFP4 cache,
 * E4M3 window, bf16 query/output.
 */
int csa2_sparse_attn_layers(const csa2_params* p, int L, int B,
                            const void* q, const float* sink,
                            const void* const* win, const int32_t* n_tokens,
                            const void* const* comp, const uint8_t* const* comp_scales,
                            const int32_t* idx, void* out,
                            int32_t* dev_status, void* stream);

/*
 * csa2_sparse_attn_layers_part — csa2_sparse_attn_layers restricted to the
 * sequences [b0, b0 + nb) of the batch of B: all arrays keep their full-batch
 * shapes and layouts (q/out [L, B, H, D], win [L*B], n_tokens/comp/
 * comp_scales [B], idx [B, topk_pos]) and only the rows of those sequences are
 * read or written. Lets a caller pipeline micro-batches of one decode step.
 * Requires 0 <= b0, 0 <= nb, b0 + nb <= B.
 */
int csa2_sparse_attn_layers_part(const csa2_params* p, int L, int B, int b0, int nb,
                                 const void* q, const float* sink,
                                 const void* const* win, const int32_t* n_tokens,
                                 const void* const* comp, const uint8_t* const* comp_scales,
                                 const int32_t* idx, void* out,
                                 int32_t* dev_status, void* stream);

/*
 * csa2_sparse_attn_layers_split — csa2_sparse_attn_layers with the work spread
 * evenly over the CTAs. ("DeepSeek-V4.1-Flash-NVFP4" §3.4: the pages' kernel
 * splits the positions of a query across CTAs and merges the parts by their
 * log-sum-exp; here only units cut by a CTA boundary are split.)
 * The L*B units x 5 tiles of 128 positions (idx in 128s, then the window) are cut
 * into one contiguous range of equal length per CTA (one CTA per SM, or
 * p->max_ctas), so no SM idles while others finish a third unit. A unit cut by
 * a range boundary is computed in two pieces; each piece leaves its partial
 * (unnormalised O, running maximum and sum per head) in its boundary's slot of
 * the workspace and the piece that finishes second merges both and writes out.
 * Arguments and results as csa2_sparse_attn_layers, plus:
 *   workspace: device memory of at least
 *     csa2_sparse_attn_layers_split_workspace_size(p, L, B) bytes, 256-byte
 *     aligned, ZERO-FILLED before its first use (it holds one completion count
 *     per boundary, which every launch that completes leaves at zero again).
 *     Launches that share a workspace must be ordered (one stream or events).
 *     After a launch that raised CSA2_DEV_TIMEOUT, zero it again.
 *   A smaller or NULL workspace returns CSA2_ERR_INVALID_ARG (nothing enqueued);
 *   a misaligned one CSA2_ERR_ALIGN.
 */
int csa2_sparse_attn_layers_split(const csa2_params* p, int L, int B,
                                  const void* q, const float* sink,
                                  const void* const* win, const int32_t* n_tokens,
                                  const void* const* comp, const uint8_t* const* comp_scales,
                                  const int32_t* idx, void* out,
                                  void* workspace, size_t ws_bytes,
                                  int32_t* dev_status, void* stream);

/*
 * Workspace bytes of csa2_sparse_attn_layers_split for L layers x B sequences
 * on the CURRENT device (its SM count and p->max_ctas fix the grid): one
 * 263,168-byte slot per CTA boundary (about 40 MB at 152 SMs) plus the counts.
 * 0 for empty sizes or a NULL p.
 */
size_t csa2_sparse_attn_layers_split_workspace_size(const csa2_params* p, int L, int B);

/*
 * csa2_sparse_attn_layers_mma — the same contract as csa2_sparse_attn_layers on
 * the legacy warp-level tensor-core path (mma.sync bf16, P rounded to bf16),
 * one CTA per (layer, sequence) with the output accumulator in registers.
 * Kept as a second, independent implementation of the fused reader attention.
 */
int csa2_sparse_attn_layers_mma(const csa2_params* p, int L, int B,
                                const void* q, const float* sink,
                                const void* const* win, const int32_t* n_tokens,
                                const void* const* comp, const uint8_t* const* comp_scales,
                                const int32_t* idx, void* out,
                                int32_t* dev_status, void* stream);

/*
 * csa2_sparse_attn_noalloc — csa2_sparse_attn without a caller workspace.
 * (No counterpart in the pages: an addition for callers that cannot allocate.)
 *
 * Some callers cannot allocate device memory: a serving engine that has already
 * given the free HBM to its own pool (the KV cache is sized to fill it), or a
 * latency-critical path where cudaMalloc/cudaFree would synchronise the device.
 * This entry point allocates nothing: its scratch is a fixed array inside the
 * library (21,053,440 bytes, enough for 32 sequences), held on every GPU that
 * loads the library until the process exits. Arguments, results and kernels are
 * those of csa2_sparse_attn, minus workspace/ws_bytes.
 *   - B > 32 returns CSA2_ERR_UNSUPPORTED (nothing enqueued): split the batch.
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream
 *     capture.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents (nothing in it needs clearing between calls). Calls whose kernels
 *     overlap on the GPU (different streams, no ordering between them) race on
 *     it: order them on one stream or with events.
 */
int csa2_sparse_attn_noalloc(const csa2_params* p, int B,
                             const void* q, const float* sink,
                             const void* const* win, const int32_t* n_tokens,
                             const void* const* comp, const uint8_t* const* comp_scales,
                             const int32_t* idx, void* out,
                             int32_t* dev_status, void* stream);

/*
 * csa2_fp4_mma_peak — measurement aid, no counterpart in the pages: the rate of
 * the block-scaled FP4 tensor-core MMA that csa2_index_scores_shared issues, so
 * its throughput can be quoted as a fraction of what the GPU reaches with the
 * same instruction. Launches `ctas` CTAs; each issues `iters` pairs of
 * tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (M = N = 128, K = 64 each)
 * back to back from shared-memory operands into one TMEM accumulator:
 * 2 x 128 x 128 x 128 flop per pair and CTA. The caller times the launch (CUDA
 * events on `stream`). Nothing is read or written outside the kernel except
 * dev_status (CSA2_DEV_TIMEOUT if the completion wait gave up; may be NULL).
 * Requires 1 <= ctas <= 65535, 1 <= iters <= 2^22 (else CSA2_ERR_INVALID_ARG).
 */
int csa2_fp4_mma_peak(int ctas, int iters, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
