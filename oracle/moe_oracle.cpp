/*
 * CPU oracle for the 4-bit groupwise-affine MoE layer.  TEST INFRASTRUCTURE
 * ONLY: loaded by the tests, the smoke check and the benchmark's CPU-baseline
 * leg, never by the product path.  See moe_oracle.h for the page names.
 *
 * Everything is the plain definition written out, in fp64, single-threaded,
 * with no blocking, fusion or reordering: the method computes exactly a dense
 * MoE layer (only faster), so its oracle is that layer.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define GROUP 64

double oracle_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, 8 exponent bits),
 * ties to even, in one step (no detour through float). */
uint16_t oracle_double_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) */
  int quantum = e - 8;         /* 8 significant bits */
  if (quantum < -133) quantum = -133; /* bf16 subnormal spacing is 2^-133 */
  double r = nearbyint(ldexp(a, -quantum)); /* default mode: nearest, ties to even */
  double v = ldexp(r, quantum);
  if (v > 3.3895313892515355e38) return sign | 0x7F80; /* overflow to infinity */
  float f = (float)v;          /* exact: at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* [Lily-blog] "Prefill: keep routing on the GPU, dequantize in flight": every
 * group of 64 weights shares a bf16 scale and bias; [Lily-news]: the compressed
 * values carry a scale and bias used to reconstruct them.  w = q*scale + bias.
 * [DGemma] "The physics ceiling: why 300+ tok/s is blocked" proposes the same
 * groupwise format with 2-3 bit codes; here 2- and 3-bit codes are packed like
 * the 4-bit ones, low bits first along K. */
double oracle_dequant(const oracle_qmat* m, int N, int K, int e, int n, int k) {
  const int bits = m->bits ? m->bits : 4;
  /* a row's codes are one bit stream, low bits first: code k starts at bit
   * bits*k (K*bits/32 words per row; a 3-bit code may straddle two words) */
  const size_t row = (size_t)e * N + n;
  const uint32_t* words = m->q + row * (size_t)(K / 32 * bits);
  const size_t bit = (size_t)bits * (size_t)k;
  uint64_t window = words[bit / 32];
  if (bit % 32 + (size_t)bits > 32) window |= (uint64_t)words[bit / 32 + 1] << 32;
  const uint32_t code = (uint32_t)(window >> (bit % 32)) & ((1u << bits) - 1u);
  size_t g = row * (K / GROUP) + k / GROUP;
  return (double)code * oracle_bf16_to_double(m->scale[g]) + oracle_bf16_to_double(m->bias[g]);
}

void oracle_dequant_matrix(const oracle_qmat* m, int N, int K, int e, double* out) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) out[(size_t)n * K + k] = oracle_dequant(m, N, K, e, n, k);
}

/* [Lily-blog] "Why Qwen3.6-35B-A3B is a weird workload": the router scores
 * every expert for a token.  The score is the dot product of the token's
 * hidden state with the expert's router row, summed in index order. */
void oracle_router_logits(const uint16_t* X, int T, int d, const uint16_t* Wr, int E, double* logits) {
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += oracle_bf16_to_double(X[(size_t)t * d + i]) * oracle_bf16_to_double(Wr[(size_t)e * d + i]);
      logits[(size_t)t * E + e] = acc;
    }
}

typedef struct {
  float v;
  int32_t i;
} wide_entry;

/* Descending value, then ascending index; -0.0 and +0.0 compare equal. */
static int wide_cmp(const void* pa, const void* pb) {
  const wide_entry* a = (const wide_entry*)pa;
  const wide_entry* b = (const wide_entry*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->i > b->i) - (a->i < b->i);
}

/* [DGemma] "The optimizations that worked", item 1: the K best candidates of a
 * position's logits.  Written as the plain definition: sort the whole row. */
int oracle_topk_wide(const float* logits, int T, int V, int K, float* values, int32_t* indices) {
  if (T < 0 || K < 1 || V < K) return -1;
  wide_entry* row = (wide_entry*)malloc((size_t)V * sizeof(wide_entry));
  if (!row) return -1;
  for (int t = 0; t < T; ++t) {
    for (int i = 0; i < V; ++i) {
      const float v = logits[(size_t)t * V + i];
      if (isnan(v)) {
        free(row);
        return -1;
      }
      row[i].v = v;
      row[i].i = i;
    }
    qsort(row, (size_t)V, sizeof(wide_entry), wide_cmp);
    for (int j = 0; j < K; ++j) {
      values[(size_t)t * K + j] = row[j].v;
      indices[(size_t)t * K + j] = row[j].i;
    }
  }
  free(row);
  return 0;
}

typedef struct {
  float v;
  int i;
} kv;

/* Descending value; among equal values the lower index first. */
static int kv_cmp(const void* pa, const void* pb) {
  const kv* a = (const kv*)pa;
  const kv* b = (const kv*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->i > b->i) - (a->i < b->i);
}

/* [Lily-blog] "Why Qwen3.6-35B-A3B is a weird workload": a router scores the
 * experts and picks 8 of 256.  Selection is on the raw fp32 logits (softmax is
 * monotone, so membership is the same as on probabilities: the argument of
 * [DGemma] "Hierarchical exact top-K sampler chain").  The weights are the
 * softmax over E renormalised over the selected k, which equals the softmax
 * over the selected k: w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max),
 * evaluated in fp64, summed in selection order, rounded once to fp32. */
int oracle_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w) {
  if (T < 0 || E < 1 || k < 1 || k > E) return -1;
  kv* row = (kv*)malloc(sizeof(kv) * (size_t)E);
  double* ex = (double*)malloc(sizeof(double) * (size_t)k);
  if (!row || !ex) {
    free(row);
    free(ex);
    return -1;
  }
  int rc = 0;
  for (int t = 0; t < T && rc == 0; ++t) {
    for (int e = 0; e < E; ++e) {
      float v = logits[(size_t)t * E + e];
      if (!isfinite(v)) rc = -1;
      row[e].v = v;
      row[e].i = e;
    }
    if (rc) break;
    qsort(row, (size_t)E, sizeof(kv), kv_cmp);
    double top = (double)row[0].v;
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      ex[j] = exp((double)row[j].v - top);
      sum += ex[j];
    }
    for (int j = 0; j < k; ++j) {
      ids[(size_t)t * k + j] = row[j].i;
      w[(size_t)t * k + j] = (float)(ex[j] / sum);
    }
  }
  free(row);
  free(ex);
  return rc;
}

/* [Lily-blog] "Prefill: keep routing on the GPU, dequantize in flight": grouped
 * GEMM needs each expert's rows stored together, hence histogram, prefix scan,
 * scatter and block map after every top-k selection.  [Lily-news]: block size
 * adapts to each expert's row count.  Stability: within an expert, rows are in
 * ascending flattened assignment index a = t*k + j. */
int oracle_route_layout(const int32_t* ids, int T, int E, int k, int block_rows,
                        int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                        int32_t* block_map, int32_t* num_blocks) {
  if (T < 0 || E < 1 || k < 1 || block_rows < 1) return -1;
  int A = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int a = 0; a < A; ++a) {
    int e = ids[a];
    if (e < 0 || e >= E) return -1;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  if (!cursor) return -1;
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int a = 0; a < A; ++a) {
    int pos = cursor[ids[a]]++;
    perm[pos] = a;
    inv_perm[a] = pos;
  }
  free(cursor);
  int nb = 0;
  for (int e = 0; e < E; ++e) {
    for (int r = 0; r < counts[e]; r += block_rows) {
      int rows = counts[e] - r < block_rows ? counts[e] - r : block_rows;
      block_map[3 * nb + 0] = e;
      block_map[3 * nb + 1] = offsets[e] + r;
      block_map[3 * nb + 2] = rows;
      ++nb;
    }
  }
  *num_blocks = nb;
  return 0;
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* One expert on one token.  [Lily-blog] "Decode: minimize bytes per token",
 * third item: the expert input projections are followed by the gate activation
 * (SwiGLU: h = silu(gate) * up), and the output projection maps h back to d. */
void oracle_expert_apply(const uint16_t* x, int d, int I, const oracle_experts* ex, int e, double* y) {
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  if (!h) return;
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < d; ++c) {
      double xc = oracle_bf16_to_double(x[c]);
      g += oracle_dequant(&ex->gate, I, d, e, i, c) * xc;
      u += oracle_dequant(&ex->up, I, d, e, i, c) * xc;
    }
    h[i] = silu(g) * u;
  }
  for (int n = 0; n < d; ++n) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += oracle_dequant(&ex->down, d, I, e, n, i) * h[i];
    y[n] = acc;
  }
  free(h);
}

/* [Lily-blog] "Decode: minimize bytes per token", third item: the expert output
 * projection is combined with the routing scores and the shared expert;
 * [Lily-news]: one shared expert is used for every input (weight 1, no gate).
 * Y[t] = sum_j w[t][j] * expert_{ids[t][j]}(x_t) + shared(x_t). */
int oracle_forward(const uint16_t* X, int T, int d, int I, int k,
                   const oracle_experts* routed, const oracle_experts* shared, int I_shared,
                   const int32_t* ids, const float* w, int t_begin, int t_end,
                   double* Y64, uint16_t* Y16) {
  if (t_begin < 0 || t_end > T || t_begin > t_end || d < 1 || I < 1 || k < 1) return -1;
  double* y = (double*)malloc(sizeof(double) * (size_t)d);
  double* acc = (double*)malloc(sizeof(double) * (size_t)d);
  if (!y || !acc) {
    free(y);
    free(acc);
    return -1;
  }
  int rc = 0;
  for (int t = t_begin; t < t_end; ++t) {
    const uint16_t* x = X + (size_t)t * d;
    for (int n = 0; n < d; ++n) acc[n] = 0.0;
    for (int j = 0; j < k; ++j) {
      int e = ids[(size_t)t * k + j];
      if (e < 0 || e >= routed->n_experts) {
        rc = -1;
        break;
      }
      double wj = (double)w[(size_t)t * k + j];
      oracle_expert_apply(x, d, I, routed, e, y);
      for (int n = 0; n < d; ++n) acc[n] += wj * y[n];
    }
    if (rc) break;
    if (shared) {
      oracle_expert_apply(x, d, I_shared, shared, 0, y);
      for (int n = 0; n < d; ++n) acc[n] += y[n];
    }
    size_t row = (size_t)(t - t_begin) * d;
    for (int n = 0; n < d; ++n) {
      Y64[row + n] = acc[n];
      if (Y16) Y16[row + n] = oracle_double_to_bf16(acc[n]);
    }
  }
  free(y);
  free(acc);
  return rc;
}
