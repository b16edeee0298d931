// Top-k selection and routing weights for one token, by one warp.  Used by the
// routing kernel and by the decode kernel when it routes its own tokens, so
// both produce the same bits.
//
// "Perplexity's Lily Beats MLX-LM on MacBook M5", section "Why Qwen3.6-35B-A3B
// is a weird workload": the router scores 256 experts and picks 8.  Selection
// is on the raw fp32 logits (softmax is monotone); a lower expert index wins a
// tie; the weights are the softmax over the selected logits, computed in fp64
// (exp(l_j - l_max), summed in selection order) and rounded once to fp32.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace bm {

// Selection.  row: E <= 32 * kPL fp32 logits.  On return lane j < k holds the
// j-th selected expert (descending logit) in sel_i and its logit in sel_v;
// every lane learns whether the row was all finite.
template <int kPL>
__device__ __forceinline__ void warp_topk_select(const float* __restrict__ row, int E, int k, int lane, int& sel_i,
                                                 float& sel_v, bool& all_finite) {
  // Monotone 32-bit keys: a larger float gives a larger unsigned key.  -0.0
  // becomes +0.0 first, so equal floats always get equal keys.
  uint32_t key[kPL];
  uint32_t taken = 0;
  bool finite = true;
#pragma unroll
  for (int c = 0; c < kPL; ++c) {
    const int e = lane + 32 * c;
    const bool in = e < E;
    float v = in ? __ldg(row + e) : 0.0f;
    finite &= !in || isfinite(v);
    if (v == 0.0f) v = 0.0f;
    const uint32_t u = __float_as_uint(v);
    key[c] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    if (!in) taken |= 1u << c;
  }
  all_finite = __all_sync(0xffffffffu, finite);

  uint32_t sel_key = 0;  // lane j keeps the j-th selected key
  sel_i = 0;
  for (int j = 0; j < k; ++j) {
    // lane-local best: largest key, lowest index among equal keys
    uint32_t bk = 0;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int c = 0; c < kPL; ++c) {
      if (!((taken >> c) & 1u) && (key[c] > bk || bi == 0x7FFFFFFF)) {
        bk = key[c];
        bi = lane + 32 * c;
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bi == 0x7FFFFFFF ? 0u : bk);
    const int win = static_cast<int>(
        __reduce_min_sync(0xffffffffu, (bi != 0x7FFFFFFF && bk == kmax) ? static_cast<uint32_t>(bi) : 0xFFFFFFFFu));
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
    if (lane == j) {
      sel_key = kmax;
      sel_i = win;
    }
  }
  // back from key to float
  const uint32_t su = (sel_key & 0x80000000u) ? (sel_key & 0x7FFFFFFFu) : ~sel_key;
  sel_v = __uint_as_float(su);
}

// Weights of a selection (sel_v of lanes 0..k-1, lane 0 the largest): the
// softmax over the selected logits in fp64, summed in selection order, rounded
// once to fp32.  Lane j < k receives weight j.
__device__ __forceinline__ float warp_topk_weights(float sel_v, int k, int lane) {
  const float top = __shfl_sync(0xffffffffu, sel_v, 0);
  const double ex = (lane < k) ? exp(static_cast<double>(sel_v) - static_cast<double>(top)) : 0.0;
  double sum = 0.0;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
  return static_cast<float>(ex / sum);
}

}  // namespace bm
