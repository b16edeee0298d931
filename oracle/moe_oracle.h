/*
 * CPU oracle for the 4-bit groupwise-affine mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library) never calls it and shares no code with it.
 *
 * Plain, single-threaded C++ (C-style, exported with C linkage) with fp64
 * arithmetic.  Each function states the passage of the source pages it
 * follows:
 *   [Lily-news]  "Perplexity builds a custom engine for Qwen on M5 Macs"
 *   [Lily-blog]  "Perplexity's Lily Beats MLX-LM on MacBook M5. Because It Only
 *                Runs One Model." (sections named in each comment)
 *   [Lily-feed]  "Perplexity Open Sources Lily: A Rust + Metal Inference Engine
 *                for Qwen3.6-35B-A3B on Apple Silicon"
 *   [DGemma]     "Squeezing a 26B diffusion LLM onto a Mac"
 *
 * Weight layout (row-major, little-endian), b = bits per code (4, 3 or 2):
 *   q     uint32 [E][N][K*b/32]  each row one bit stream, low bits first:
 *                                the code of column k starts at bit b*k (b = 4:
 *                                bits 4*(k%8) of word k/8; b = 3: a code may
 *                                straddle two words)
 *   scale uint16 [E][N][K/64] bf16 bit patterns, one per 64-column group
 *   bias  uint16 [E][N][K/64] bf16 bit patterns
 * gate/up: N = I, K = d.  down: N = d, K = I.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  const uint32_t* q;
  const uint16_t* scale;
  const uint16_t* bias;
  int bits; /* bits per code: 4, 3 or 2 (0 means 4) */
} oracle_qmat;

typedef struct {
  oracle_qmat gate, up, down;
  int n_experts;
} oracle_experts;

/* bf16 <-> double.  oracle_double_to_bf16 rounds once, to nearest, ties to even. */
double oracle_bf16_to_double(uint16_t h);
uint16_t oracle_double_to_bf16(double x);

/* One dequantised weight: w = q * scale + bias of its group (exact in fp64),
 * q the code of m->bits bits. */
double oracle_dequant(const oracle_qmat* m, int N, int K, int e, int n, int k);

/* Dequantise a whole [N][K] matrix of expert e into out (row-major). */
void oracle_dequant_matrix(const oracle_qmat* m, int N, int K, int e, double* out);

/* Router projection: logits[t][e] = sum_i X[t][i] * Wr[e][i] in fp64 over the
 * exact bf16 values.  X uint16 [T][d], Wr uint16 [E][d] (bf16 bit patterns),
 * logits double [T][E].  [Lily-blog] "Why Qwen3.6-35B-A3B is a weird
 * workload": a router scores the 256 experts of each token; read here as a
 * linear map of the token's hidden state. */
void oracle_router_logits(const uint16_t* X, int T, int d, const uint16_t* Wr, int E, double* logits);

/* Exact top-K of each row of a wide score matrix: values [T][K] and indices
 * [T][K] of the K largest entries of logits [T][V], in descending order, a lower
 * index first among equal values (-0.0 equals +0.0).  [DGemma] "The
 * optimizations that worked", item 1: the sampler needs only the top ~64 of
 * 262,144 logits per position.  The plain definition: a full sort of each row.
 * Returns 0, or -1 on a NaN or bad sizes (1 <= K <= V). */
int oracle_topk_wide(const float* logits, int T, int V, int K, float* values, int32_t* indices);

/* Router top-k and renormalised weights.  Returns 0, or -1 on a non-finite logit
 * or bad sizes.  ids/w are [T][k], ids in selection order (descending logit,
 * lower expert index first among equal logits). */
int oracle_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w);

/* Histogram, exclusive scan, stable scatter and tile block map for ids [T*k].
 * counts [E], offsets [E+1], perm/inv_perm [T*k], block_map [max_blocks][3] as
 * (expert, first permuted row, rows).  Returns 0 or -1. */
int oracle_route_layout(const int32_t* ids, int T, int E, int k, int block_rows,
                        int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                        int32_t* block_map, int32_t* num_blocks);

/* One expert on one token: h = silu(x Wg^T) * (x Wu^T), y = h Wd^T.  y [d]. */
void oracle_expert_apply(const uint16_t* x, int d, int I, const oracle_experts* ex, int e, double* y);

/* The layer for tokens [t_begin, t_end):
 *   Y[t] = sum_j w[t][j] * expert_{ids[t][j]}(x_t) + shared(x_t)
 * Y64 [t_end-t_begin][d] in fp64; Y16 (nullable) the same rounded once to bf16.
 * shared may be NULL (no shared expert).  Returns 0 or -1. */
int oracle_forward(const uint16_t* X, int T, int d, int I, int k,
                   const oracle_experts* routed, const oracle_experts* shared, int I_shared,
                   const int32_t* ids, const float* w, int t_begin, int t_end,
                   double* Y64, uint16_t* Y16);

#ifdef __cplusplus
}
#endif
#endif
