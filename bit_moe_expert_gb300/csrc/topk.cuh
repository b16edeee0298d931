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

// Monotone 32-bit key of a logit: a larger float gives a larger unsigned key;
// -0.0 becomes +0.0 first, so equal floats always get equal keys.
__device__ __forceinline__ uint32_t topk_key(float v) {
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float topk_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Lane l's eight logits 8l .. 8l+7 of a row of E <= 256 (zero past E).
__device__ __forceinline__ void topk_load_row8(const float* __restrict__ row, int E, int lane, float (&xv)[8]) {
  if (E == 256 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    // two 16-byte loads per lane: the warp reads the row as eight whole lines
    const float4 lo = __ldcg(reinterpret_cast<const float4*>(row) + 2 * lane);
    const float4 hi = __ldcg(reinterpret_cast<const float4*>(row) + 2 * lane + 1);
    xv[0] = lo.x, xv[1] = lo.y, xv[2] = lo.z, xv[3] = lo.w;
    xv[4] = hi.x, xv[5] = hi.y, xv[6] = hi.z, xv[7] = hi.w;
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c) xv[c] = 8 * lane + c < E ? __ldcg(row + 8 * lane + c) : 0.0f;
  }
}

// Selection for E <= 256 from the lanes' loaded logits: lane l holds experts
// 8l .. 8l+7 as 64-bit values (key << 32 | ~expert), so a larger value is a
// larger logit or, for equal logits, a lower expert; it sorts them once (a
// 19-comparator network), and each of the k rounds takes the largest head key
// over the lanes (the lowest lane among equal heads holds the lowest expert,
// lanes holding contiguous experts) and pops that lane's head.
__device__ __forceinline__ void warp_topk_select_sorted_vals(const float (&xv)[8], int E, int k, int lane,
                                                             int& sel_i, float& sel_v, bool& all_finite) {
  uint64_t v[8];
  bool finite = true;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int e = 8 * lane + c;
    finite &= e >= E || isfinite(xv[c]);
    v[c] = e < E ? (static_cast<uint64_t>(topk_key(xv[c])) << 32) | static_cast<uint32_t>(~e) : 0ull;
  }
  all_finite = __all_sync(0xffffffffu, finite);
  constexpr int kNet[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6}, {5, 7}, {1, 2}, {5, 6},
                               {0, 4}, {1, 5}, {2, 6}, {3, 7}, {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
  for (int c = 0; c < 19; ++c) {
    const uint64_t a = v[kNet[c][0]], b = v[kNet[c][1]];
    v[kNet[c][0]] = a > b ? a : b;
    v[kNet[c][1]] = a > b ? b : a;
  }
  uint32_t sel_key = 0;
  sel_i = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t hk = static_cast<uint32_t>(v[0] >> 32);
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, hk);
    const unsigned cand = __ballot_sync(0xffffffffu, hk == kmax && v[0] != 0ull);
    const int win = __ffs(cand) - 1;
    const uint32_t wlow = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v[0]), win);
    if (lane == j) {
      sel_key = kmax;
      sel_i = static_cast<int>(~wlow);
    }
    if (lane == win) {
#pragma unroll
      for (int c = 0; c < 7; ++c) v[c] = v[c + 1];
      v[7] = 0ull;
    }
  }
  sel_v = topk_key_value(sel_key);
}

__device__ __forceinline__ void warp_topk_select_sorted(const float* __restrict__ row, int E, int k, int lane,
                                                        int& sel_i, float& sel_v, bool& all_finite) {
  float xv[8];
  topk_load_row8(row, E, lane, xv);
  warp_topk_select_sorted_vals(xv, E, k, lane, sel_i, sel_v, all_finite);
}

// Selection.  row: E <= 32 * kPL fp32 logits.  On return lane j < k holds the
// j-th selected expert (descending logit) in sel_i and its logit in sel_v;
// every lane learns whether the row was all finite.
template <int kPL>
__device__ __forceinline__ void warp_topk_select(const float* __restrict__ row, int E, int k, int lane, int& sel_i,
                                                 float& sel_v, bool& all_finite) {
  if constexpr (kPL == 8) {
    warp_topk_select_sorted(row, E, k, lane, sel_i, sel_v, all_finite);
    return;
  }
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
