/*
 * CSA2 CPU oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 restatement of the per-layer CSA2 path (Compressor ->
 * NVFP4 cache -> Indexer -> two-level top-k -> sparse attention with sink).
 * Only the test suite, the smoke check and the bench's CPU-baseline leg may
 * load this library. The product (the CUDA library) never links or calls it,
 * and this file shares no code, header, table or constant with it.
 *
 * Sources (page title, section):
 *   [NVFP4]  "DeepSeek-V4.1-Flash-NVFP4" walkthrough (lpnh.cn):
 *            §三 (layer diagram: 128 window + 512 compressed = 640 per query),
 *            §3.1 (128-token FP8 ring window), §3.2 (2:1 softmax-gated
 *            Compressor, NVFP4 = 16-element groups with an E4M3 scale),
 *            §3.3 (Indexer: 32 FP4 index heads, ReLU, per-head weights;
 *            blocks of 8, top-2048 blocks with the newest kept, top-512
 *            positions), §3.4 (sparse_attn: gather, online softmax, attn_sink),
 *            §四 (memory ledger).
 *   [CFG]    "CSA2稀疏注意力、384专家MoE与1M上下文" config walkthrough (nxmr.cn),
 *            §2.1 (index_n_heads 32, index_head_dim 128, index_topk 512,
 *            candidate_block_size 8, candidate_topk_blocks 2048,
 *            sliding_window 128), §一 (64 Q heads / 1 KV head).
 *
 * Every function below is single-threaded and re-entrant (no global state).
 * Parity status of each function is stated in its comment; all are pinned by
 * the CPU test suite (tests/test_oracle_*.py).
 */
#ifndef CSA2_ORACLE_H
#define CSA2_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ([NVFP4] §3.2: E2M1 values, E4M3 group scales; §3.1 FP8 window) ---- */
/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa; code in 0..15.            */
double orc_e2m1_value(int code);
/* E4M3 ("fn": no infinities, S.1111.111 = NaN): 1 sign, 4 exp (bias 7), 3 mantissa. */
double orc_e4m3_value(int code);
/* Nearest E4M3 value to x, ties to even code, |x| > 448 saturates to 448.   */
int orc_e4m3_encode(float x);
/* Nearest E2M1 value to x, ties to even code, |x| > 6 saturates to 6;
 * the sign bit follows the sign of x (so -0 and tiny negatives give 0x8).   */
int orc_e2m1_encode(float x);

/* NVFP4 quantisation of n_groups groups of 16 fp32 values ([NVFP4] §3.2):
 *   amax = max|x|, s = fl32(amax/6), S = E4M3(s), code_i = E2M1(fl32(x_i/S)),
 *   S == 0 gives all-zero codes. Element 2k -> low nibble of byte k.
 *   vals: 8 bytes per group, scales: 1 byte per group.                     */
void orc_nvfp4_quantize(const float* x, int64_t n_groups, uint8_t* vals, uint8_t* scales);
/* Value of element i of an NVFP4 row (vals + one scale per 16 elements).    */
double orc_nvfp4_value(const uint8_t* vals, const uint8_t* scales, int64_t i);

/* ---- Compressor ([NVFP4] §3.2) ---- */
/* Softmax-gated pool of one channel of a token pair, rounded to fp32.       */
float orc_pool(float kv0, float kv1, float g0, float g1);

/*
 * One Compressor/window append for ONE sequence ([NVFP4] §3.1, §3.2).
 * State: T raw tokens seen so far; if T is odd, pend_kv/pend_g hold token T-1.
 * Appends n_new tokens (rows of D channels in kv_new/g_new):
 *   - every completed pair j (tokens 2j, 2j+1) is pooled and written to
 *     compressed row j: NVFP4 (comp_vals [.,D/2] + comp_scales [.,D/16]) when
 *     comp_f32 == NULL, else fp32 rows in comp_f32 [., D];
 *   - every new raw token p writes ring slot p mod W of the window:
 *     E4M3 bytes in win_u8 [W, D] or fp32 in win_f32 [W, D] (one is non-NULL;
 *     both NULL means "no window");
 *   - comp_vals/comp_scales/comp_f32 all NULL means a window-only layer.
 * Returns the new T.                                                        */
int64_t orc_compress_append(int64_t T, int n_new, int D, int W,
                            const float* kv_new, const float* g_new,
                            float* pend_kv, float* pend_g,
                            uint8_t* comp_vals, uint8_t* comp_scales, float* comp_f32,
                            uint8_t* win_u8, float* win_f32);

/* The same for a layer of compression ratio 1 or 2. Ratio 1 (the uncompressed
 * 1:1 layers, [CFG] §2.2, [NVFP4] §3.2): pooling is skipped, raw token p is
 * quantized (or copied, fp32) into compressed row p; gate and pending state are
 * unused. Ratio 2 is orc_compress_append. */
int64_t orc_compress_append_ratio(int64_t T, int n_new, int D, int W, int ratio,
                                  const float* kv_new, const float* g_new,
                                  float* pend_kv, float* pend_g,
                                  uint8_t* comp_vals, uint8_t* comp_scales, float* comp_f32,
                                  uint8_t* win_u8, float* win_f32);

/* ---- Rotary position embedding of the compressed KV ---- */
/*
 * [CFG] §2.2 (compress_rope_theta 160000: the compressed KV gets its own RoPE
 * base), §四 (rope_scaling: rope_type yarn, factor 16,
 * original_max_position_embeddings 65536, beta_fast 32, beta_slow 1);
 * [NVFP4] §3.2 (one latent stands for 2 tokens, so it uses compress_rope_theta
 * 160000 with YaRN factor 16 to reach 1M).
 * Method: RoPE as in Su et al., "RoFormer" (2021) — dims (2i, 2i+1) of the
 * rotated part turn by the angle pos * theta_i, theta_i = base^(-2i/dim) —
 * with YaRN's "NTK-by-parts" frequencies (Peng et al., "YaRN", 2023): with
 * wavelength lambda_i = 2 pi / theta_i and r_i = orig_len / lambda_i, a pair
 * with r_i > beta_fast keeps theta_i, one with r_i < beta_slow takes
 * theta_i / factor, and between them gamma = (r_i - beta_slow) /
 * (beta_fast - beta_slow) blends (1 - gamma) theta_i / factor + gamma theta_i.
 * Readings (the pages name only the base and the YaRN keys): the rotated part
 * is the last `dim` dims of the latent; compressed row j sits at raw position
 * ratio * j (the first raw token of its pair); YaRN's attention temperature is
 * a logit scale, not part of the rotation.
 */
typedef struct orc_rope {
    int dim;           /* rotated dims (even): the last `dim` of the row; 0 = none */
    double base;       /* rotary base (compress_rope_theta) */
    double factor;     /* YaRN scale s; 1 gives plain RoPE */
    double orig_len;   /* original context length L */
    double beta_fast;  /* above this many rotations over L a pair keeps its frequency */
    double beta_slow;  /* below this many it is interpolated by 1/factor */
} orc_rope;

/* theta'_i of pairs i = 0 .. dim/2-1 (fp64).                                */
void orc_rope_freqs(const orc_rope* r, double* theta);
/* Rotates x[D-dim .. D) of one fp32 row in place at raw position pos: pair i =
 * (x[D-dim+2i], x[D-dim+2i+1]) -> (a cos - b sin, a sin + b cos), angle
 * pos * theta'_i, fp64 arithmetic, rounded to fp32. NULL or dim 0: no-op.   */
void orc_rope_rotate(float* x, int D, int64_t pos, const orc_rope* r);

/* One compressed row j of a layer of compression ratio 1 or 2 ([NVFP4] §3.2):
 * kv0 (and kv1, g0, g1 at ratio 2) are the raw tokens ratio*j (.. ratio*j+1);
 * the row is the gated pool (ratio 2) or the token itself (ratio 1), rotated at
 * raw position ratio*j when rope is set, then written as NVFP4 (vals [D/2],
 * scales [D/16]) or, when f32 is non-NULL, as fp32 [D].                     */
void orc_compress_row(int D, int ratio, int64_t j, const float* kv0, const float* kv1,
                      const float* g0, const float* g1, const orc_rope* rope,
                      uint8_t* vals, uint8_t* scales, float* f32);

/* orc_compress_append_ratio with the compressed rows rotated (rope may be NULL). */
int64_t orc_compress_append_rope(int64_t T, int n_new, int D, int W, int ratio,
                                 const orc_rope* rope, const float* kv_new, const float* g_new,
                                 float* pend_kv, float* pend_g,
                                 uint8_t* comp_vals, uint8_t* comp_scales, float* comp_f32,
                                 uint8_t* win_u8, float* win_f32);

/* ---- Indexer ([NVFP4] §3.3, [CFG] §2.1) ---- */
/*
 * s_t = sum_h w[h] * ReLU( sum_d q[h,d] * k[t,d] ),  t < n_c, fp64.
 * q: Hi heads x Di dims NVFP4 (q_vals [Hi, Di/2], q_scales [Hi, Di/16]);
 * keys: n_c rows NVFP4 (k_vals [n_c, Di/2], k_scales [n_c, Di/16]).
 * scores[t] is the fp64 sum rounded to fp32. Returns the number of scores
 * that are NOT guaranteed exact: a score is exact when every product and
 * every partial sum, in any order, is representable in fp32 (all terms are
 * multiples of their smallest power-of-two granule r and sum|terms| < 2^24 r).
 */
int64_t orc_index_scores(int Hi, int Di, const uint8_t* q_vals, const uint8_t* q_scales,
                         const float* w, int64_t n_c, const uint8_t* k_vals,
                         const uint8_t* k_scales, float* scores);
/* Block maxima over blocks of `blk` positions (last block: valid ones only). */
void orc_block_max(const float* scores, int64_t n_c, int blk, float* block_max);

/* ---- Two-level selection ([NVFP4] §3.3) ---- */
/*
 * Blocks of `blk` positions scored by their max score. If there are more than
 * Kb blocks, keep the newest block (the one holding position n_c-1) and the
 * best Kb-1 of the others, ordered by (score desc, block index asc); else keep
 * all. Then among the positions of the kept blocks keep the best Kp by
 * (score desc, position asc). Writes them ascending to idx[0..Kp), pads with
 * -1, returns how many are valid.                                           */
int orc_select(const float* scores, int64_t n_c, int blk, int Kb, int Kp, int32_t* idx);

/* ---- sparse attention with sink ([NVFP4] §3.4, §三, §3.1) ---- */
/*
 * One query (H heads x D dims, fp64 values in q). The attended set is
 *   - the window: raw positions max(0,T-W)..T-1, row (p mod W) of the ring
 *     (win_u8 E4M3 bytes or win_f32 fp32 rows; both NULL = no window);
 *   - the compressed rows idx[0..n_idx) that are >= 0, from comp_vals/
 *     comp_scales (NVFP4) or comp_f32 (fp32).
 * z_j = scale * q_h . k_j ; out_h = sum_j e^{z_j} v_j / (e^{sink_h} + sum_j e^{z_j}),
 * with K = V = the stored latent. Two-pass softmax in fp64. out: H x D.
 * Returns the number of attended positions.                                 */
int orc_sparse_attn(int H, int D, const double* q, const double* sink, double scale,
                    int64_t T, int W, const uint8_t* win_u8, const float* win_f32,
                    const uint8_t* comp_vals, const uint8_t* comp_scales, const float* comp_f32,
                    const int32_t* idx, int n_idx, double* out);

/* ---- closed forms from the memory ledger ([NVFP4] §四, §3.1, §一, §三) ---- */
/* Bytes of NVFP4 payload / E4M3 scales for n positions of D channels.      */
int64_t orc_nvfp4_payload_bytes(int64_t n, int D);
int64_t orc_nvfp4_scale_bytes(int64_t n, int D);

#ifdef __cplusplus
}
#endif
#endif
