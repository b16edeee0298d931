// Decode path (small T): the expert projections as matrix-vector products on
// the CUDA cores.  "Perplexity's Lily Beats MLX-LM on MacBook M5", section
// "Prefill and decode are different problems": batch-1 decode is a GEMV bound
// by memory bandwidth that belongs on the vector ALUs; section "Decode:
// minimize bytes per token": the expert input projections are fused with the
// gate activation, and the output projection with the routing scores and the
// shared expert.
//
// Design (sm_103a): one cooperative launch per layer, one CTA per SM.
//   phase 1  each CTA owns a tile of 32 rows of gate and up of one (token,
//            expert) pair: h = silu(x Wg^T) * (x Wu^T) for those rows -> global
//   barrier  a grid-wide barrier (bounded wait)
//   phase 2  each CTA owns 16 output rows of one token: the down projection of
//            every selected expert and the shared expert, weighted and summed
//            -> Y (bf16)
// Every CTA issues, up front, TMA loads of all the weight bytes of BOTH its
// tiles -- codes and group parameters -- so each active expert's bytes cross
// HBM exactly once and the down-projection weights stream in while phase 1
// computes.  A thread owns a row and a slice of K; the activation vector is
// broadcast from shared memory.  The 4-bit codes become fp32 values 128+q with
// one byte permute each (exponent of 128, code in the low mantissa bits), are
// multiplied by x with packed fp32x2 FMAs (four independent accumulators), and
// the affine map is applied once per 64-column group:
//   sum_k (q_k s + b) x_k = s * sum_k (128+q_k) x_k + (b - 128 s) * sum_k x_k.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bm {

namespace {

constexpr int kThreads = 512;
constexpr int kR1 = kGemvRowsGU;     // phase-1 rows per tile (lane = row)
constexpr int kS1 = kThreads / 32;   // phase-1 K slices (one per warp)
constexpr int kR2 = kGemvRowsDown;   // phase-2 rows per tile
constexpr int kS2 = kThreads / kR2;  // phase-2 work slices
constexpr uint32_t kMagic128 = 0x43000000u;  // fp32 128.0: a code in bits 16..19 reads as 128 + q
constexpr int kBoxWords = 32;                // 128-byte rows per TMA box
constexpr int kBoxKB = 4;                    // 64-column groups per box row
constexpr long long kBarrierLimitCycles = 4000000000ll;

__host__ __device__ constexpr int div_up(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// sum over the 8 codes of one word of (128 + q) * x, into a pair accumulator.
__device__ __forceinline__ float2 codes_dot8(uint32_t w, float4 xa, float4 xb, float2 acc) {
  const uint32_t lo = w & 0x0F0F0F0Fu;         // codes 0, 2, 4, 6 in bytes 0..3
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // codes 1, 3, 5, 7
  const float2 q01 = make_float2(__uint_as_float(prmt(lo, kMagic128, 0x7054)),
                                 __uint_as_float(prmt(hi, kMagic128, 0x7054)));
  const float2 q23 = make_float2(__uint_as_float(prmt(lo, kMagic128, 0x7154)),
                                 __uint_as_float(prmt(hi, kMagic128, 0x7154)));
  const float2 q45 = make_float2(__uint_as_float(prmt(lo, kMagic128, 0x7254)),
                                 __uint_as_float(prmt(hi, kMagic128, 0x7254)));
  const float2 q67 = make_float2(__uint_as_float(prmt(lo, kMagic128, 0x7354)),
                                 __uint_as_float(prmt(hi, kMagic128, 0x7354)));
  acc = f32x2_fma(q01, make_float2(xa.x, xa.y), acc);
  acc = f32x2_fma(q23, make_float2(xa.z, xa.w), acc);
  acc = f32x2_fma(q45, make_float2(xb.x, xb.y), acc);
  acc = f32x2_fma(q67, make_float2(xb.z, xb.w), acc);
  return acc;
}

// One row's contribution from one 64-column group.
//   tile: the TMA box holding the row (128-byte rows, 128-byte swizzle)
//   row:  row inside the box; kb: group index (selects the 32-byte chunk pair)
//   xg:   the 64 fp32 x values of this group (shared memory, broadcast)
__device__ __forceinline__ float group_dot(const uint8_t* tile, int row, int kb, const float* xg, float sx,
                                           uint32_t sbv) {
  const int c0 = ((kb & 3) * 2) ^ (row & 7);
  const int c1 = ((kb & 3) * 2 + 1) ^ (row & 7);
  const uint4 wa = *reinterpret_cast<const uint4*>(tile + row * 128 + c0 * 16);
  const uint4 wb = *reinterpret_cast<const uint4*>(tile + row * 128 + c1 * 16);
  const float4* x4 = reinterpret_cast<const float4*>(xg);
  float2 a0 = make_float2(0.0f, 0.0f), a1 = a0, a2 = a0, a3 = a0;
  a0 = codes_dot8(wa.x, x4[0], x4[1], a0);
  a1 = codes_dot8(wa.y, x4[2], x4[3], a1);
  a2 = codes_dot8(wa.z, x4[4], x4[5], a2);
  a3 = codes_dot8(wa.w, x4[6], x4[7], a3);
  a0 = codes_dot8(wb.x, x4[8], x4[9], a0);
  a1 = codes_dot8(wb.y, x4[10], x4[11], a1);
  a2 = codes_dot8(wb.z, x4[12], x4[13], a2);
  a3 = codes_dot8(wb.w, x4[14], x4[15], a3);
  const float p = ((a0.x + a0.y) + (a1.x + a1.y)) + ((a2.x + a2.y) + (a3.x + a3.y));
  const float s = __uint_as_float(sbv << 16);
  const float b = __uint_as_float(sbv & 0xFFFF0000u);
  return fmaf(s, p, (b - 128.0f * s) * sx);
}

// Copies n floats (n % 4 == 0, 16-byte aligned) from global memory (read
// through L2) into shared memory: every load of a thread is issued before its
// first store, so the copy costs one memory latency, not one per element.
__device__ __forceinline__ void stage_f32(float* __restrict__ dst, const float* __restrict__ src, int n) {
  constexpr int kU = 8;
  const int n4 = n / 4;
  for (int base = threadIdx.x; base < n4; base += kThreads * kU) {
    float4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int f = base + u * kThreads;
      if (f < n4) v[u] = __ldcg(reinterpret_cast<const float4*>(src) + f);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int f = base + u * kThreads;
      if (f < n4) reinterpret_cast<float4*>(dst)[f] = v[u];
    }
  }
}

// bf16 [n] (n % 8 == 0, 16-byte aligned) -> fp32 in shared memory, loads first.
__device__ __forceinline__ void stage_bf16(float* __restrict__ dst, const uint16_t* __restrict__ src, int n) {
  constexpr int kU = 4;
  const int n8 = n / 8;
  for (int base = threadIdx.x; base < n8; base += kThreads * kU) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int f = base + u * kThreads;
      if (f < n8) v[u] = __ldg(reinterpret_cast<const uint4*>(src) + f);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int f = base + u * kThreads;
      if (f < n8) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        float4* d4 = reinterpret_cast<float4*>(dst + f * 8);
        d4[0] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                            __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
        d4[1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                            __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
      }
    }
  }
}

struct Layout {
  int nbox1, KB1, nbox2r, nbox2s, KB2r, KB2s, nexp, Imax;
  size_t sb1_slot, sb2_slot;
  size_t q1, sb1, x1, sx1, red1;
  size_t q2, q2s, sb2, sb2s, h2, sx2, w2, red2;
  size_t bars, total;
};

// TMA destinations start on 1024 bytes (swizzled code boxes) or 128 bytes
// (group parameters).
__host__ __device__ inline Layout layout(int d, int I, int I_shared, int k) {
  Layout L;
  L.KB1 = d / 64;
  L.nbox1 = div_up(d / 8, kBoxWords);
  L.KB2r = I / 64;
  L.KB2s = I_shared / 64;
  L.nbox2r = div_up(I / 8, kBoxWords);
  L.nbox2s = I_shared > 0 ? div_up(I_shared / 8, kBoxWords) : 0;
  L.nexp = k + (I_shared > 0 ? 1 : 0);
  L.Imax = I > I_shared ? I : I_shared;
  L.sb1_slot = round_up(static_cast<size_t>(L.KB1) * kR1 * 4, 128);
  L.sb2_slot = round_up(static_cast<size_t>(L.KB2r) * kR2 * 4, 128);
  size_t o = 0;
  L.q1 = o;
  o += 2ull * L.nbox1 * kR1 * 128;
  L.sb1 = o;
  o += 2 * L.sb1_slot;
  L.x1 = o;
  o += static_cast<size_t>(d) * 4;
  L.sx1 = o;
  o += static_cast<size_t>(L.KB1) * 4;
  o = round_up(o, 16);
  L.red1 = o;
  o += 2ull * kS1 * kR1 * 4;
  o = round_up(o, 1024);
  L.q2 = o;
  o += static_cast<size_t>(k) * L.nbox2r * kR2 * 128;
  L.q2s = o;
  o += static_cast<size_t>(L.nbox2s) * kR2 * 128;
  L.sb2 = o;
  o += static_cast<size_t>(k) * L.sb2_slot;
  L.sb2s = o;
  o += round_up(static_cast<size_t>(L.KB2s) * kR2 * 4, 128);
  L.h2 = o;  // routed h rows [k][I], then the shared expert's [I_shared]
  o += (static_cast<size_t>(k) * I + I_shared) * 4;
  L.sx2 = o;
  o += static_cast<size_t>(L.nexp) * (L.Imax / 64) * 4;
  L.w2 = o;
  o += static_cast<size_t>(L.nexp) * 4;
  o = round_up(o, 16);
  L.red2 = o;
  o += static_cast<size_t>(kS2) * kR2 * 4;
  L.bars = o;
  o += static_cast<size_t>(L.nbox1 + 1 + L.nexp) * 8;
  L.total = o + 1024;
  return L;
}

struct Tile1 {
  int pair, t, n0;
  bool shared;
};

__device__ __forceinline__ Tile1 tile1(const GemvArgs& a, int i) {
  Tile1 m;
  const int tr = a.I / kR1;
  const int routed = a.T * a.k * tr;
  if (i < routed) {
    m.pair = i / tr;
    m.n0 = (i % tr) * kR1;
    m.t = m.pair / a.k;
    m.shared = false;
  } else {
    const int ts = a.I_shared / kR1;
    const int j = i - routed;
    m.t = j / ts;
    m.n0 = (j % ts) * kR1;
    m.pair = -1;
    m.shared = true;
  }
  return m;
}

__device__ __forceinline__ int expert_of(const GemvArgs& a, int idx) {
  int e = a.ids[idx];
  if (e < 0 || e >= a.E) {
    record_status(a.status, MOE_ERR_INVALID_ARG);
    e = 0;
  }
  return e;
}

// Grid-wide barrier over all CTAs of this (cooperative) launch.  The counter is
// reset by the last arrival, which then advances the generation; a wait that
// exceeds the limit records MOE_ERR_TIMEOUT and lets the CTA continue.
__device__ __forceinline__ void grid_barrier(WsHeader* hdr, uint32_t* status) {
  __threadfence();  // every thread's global writes (h) before the arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile uint32_t* gen_p = &hdr->bar_gen;
    __threadfence();
    const uint32_t gen = *gen_p;
    const uint32_t arrived = atomicAdd(&hdr->bar_count, 1u);
    if (arrived == gridDim.x - 1) {
      atomicExch(&hdr->bar_count, 0u);
      __threadfence();
      atomicAdd(&hdr->bar_gen, 1u);
    } else {
      const long long t0 = clock64();
      while (*gen_p == gen) {
        __nanosleep(64);
        if (clock64() - t0 > kBarrierLimitCycles) {
          record_status(status, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap qg_r, const __grid_constant__ CUtensorMap qu_r,
                  const __grid_constant__ CUtensorMap sbg_r, const __grid_constant__ CUtensorMap sbu_r,
                  const __grid_constant__ CUtensorMap qd_r, const __grid_constant__ CUtensorMap sbd_r,
                  const __grid_constant__ CUtensorMap qg_s, const __grid_constant__ CUtensorMap qu_s,
                  const __grid_constant__ CUtensorMap sbg_s, const __grid_constant__ CUtensorMap sbu_s,
                  const __grid_constant__ CUtensorMap qd_s, const __grid_constant__ CUtensorMap sbd_s, GemvArgs a,
                  WsHeader* hdr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int k = a.k;
  const int K = a.d;
  const Layout L = layout(a.d, a.I, a.I_shared, k);
  const bool has_shared = a.I_shared > 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint8_t* qg = smem + L.q1;
  uint8_t* qu = qg + static_cast<size_t>(L.nbox1) * kR1 * 128;
  uint32_t* sbg = reinterpret_cast<uint32_t*>(smem + L.sb1);
  uint32_t* sbu = reinterpret_cast<uint32_t*>(smem + L.sb1 + L.sb1_slot);
  float* xs = reinterpret_cast<float*>(smem + L.x1);
  float* sxs = reinterpret_cast<float*>(smem + L.sx1);
  float* red1 = reinterpret_cast<float*>(smem + L.red1);
  uint8_t* q2 = smem + L.q2;
  uint8_t* q2s = smem + L.q2s;
  uint32_t* sb2s = reinterpret_cast<uint32_t*>(smem + L.sb2s);
  float* hs = reinterpret_cast<float*>(smem + L.h2);
  float* sx2 = reinterpret_cast<float*>(smem + L.sx2);
  float* w2 = reinterpret_cast<float*>(smem + L.w2);
  float* red2 = reinterpret_cast<float*>(smem + L.red2);
  uint64_t* bars1 = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* bars2 = bars1 + L.nbox1 + 1;
  const size_t box1 = kR1 * 128;
  const size_t box2 = kR2 * 128;

  const int n1 = a.T * k * (a.I / kR1) + (has_shared ? a.T * (a.I_shared / kR1) : 0);
  const int tiles2 = a.d / kR2;
  const int n2 = a.T * tiles2;

  if (threadIdx.x == 0) {
    for (int b = 0; b < L.nbox1 + 1 + L.nexp; ++b) mbar_init(&bars1[b], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Warp 0: lane b < nbox1 loads code box b of gate and up; lane nbox1 the group parameters.
  auto issue1 = [&](const Tile1& m, int e) {
    if (warp != 0) return;
    const CUtensorMap* mg = m.shared ? &qg_s : &qg_r;
    const CUtensorMap* mu = m.shared ? &qu_s : &qu_r;
    if (lane < L.nbox1) {
      mbar_arrive_expect_tx(&bars1[lane], static_cast<uint32_t>(2 * box1));
      tma_load_3d(qg + lane * box1, mg, &bars1[lane], lane * kBoxWords, m.n0, e);
      tma_load_3d(qu + lane * box1, mu, &bars1[lane], lane * kBoxWords, m.n0, e);
    } else if (lane == L.nbox1) {
      mbar_arrive_expect_tx(&bars1[L.nbox1], static_cast<uint32_t>(2 * L.KB1 * kR1 * 4));
      tma_load_3d(sbg, m.shared ? &sbg_s : &sbg_r, &bars1[L.nbox1], m.n0, 0, e);
      tma_load_3d(sbu, m.shared ? &sbu_s : &sbu_r, &bars1[L.nbox1], m.n0, 0, e);
    }
  };
  // Warp 1: lane j < k loads routed expert j's down rows; lane k the shared expert's.
  auto issue2 = [&](int t, int n0, bool routed_part) {
    if (warp != 1) return;
    const int j = lane;
    if (routed_part && j < k) {
      const int e = expert_of(a, t * k + j);
      uint8_t* qj = q2 + static_cast<size_t>(j) * L.nbox2r * box2;
      uint32_t* sbj = reinterpret_cast<uint32_t*>(smem + L.sb2 + static_cast<size_t>(j) * L.sb2_slot);
      mbar_arrive_expect_tx(&bars2[j], static_cast<uint32_t>(L.nbox2r * box2 + L.KB2r * kR2 * 4));
      tma_load_3d(sbj, &sbd_r, &bars2[j], n0, 0, e);
      for (int b = 0; b < L.nbox2r; ++b) tma_load_3d(qj + b * box2, &qd_r, &bars2[j], b * kBoxWords, n0, e);
    } else if (!routed_part && j == k && has_shared) {
      mbar_arrive_expect_tx(&bars2[k], static_cast<uint32_t>(L.nbox2s * box2 + L.KB2s * kR2 * 4));
      tma_load_3d(sb2s, &sbd_s, &bars2[k], n0, 0, 0);
      for (int b = 0; b < L.nbox2s; ++b) tma_load_3d(q2s + b * box2, &qd_s, &bars2[k], b * kBoxWords, n0, 0);
    }
  };
  auto routed_expert1 = [&](const Tile1& m) {
    return (!m.shared && warp == 0 && lane <= L.nbox1) ? expert_of(a, m.pair) : 0;
  };

  const int first1 = blockIdx.x;
  const int first2 = blockIdx.x;
  // Weights that do not depend on the previous kernel start streaming first.
  if (first1 < n1) {
    const Tile1 m = tile1(a, first1);
    if (m.shared) issue1(m, 0);
  }
  if (first2 < n2) issue2(first2 / tiles2, (first2 % tiles2) * kR2, false);
  pdl_wait();  // routing (and X) come from earlier kernels
  if (first1 < n1) {
    const Tile1 m = tile1(a, first1);
    if (!m.shared) issue1(m, routed_expert1(m));
  }
  if (first2 < n2) issue2(first2 / tiles2, (first2 % tiles2) * kR2, true);

  // ---------------------------------------------------------------- phase 1: h = silu(g) * u
  uint32_t par1 = 0;
  int staged_t = -1;
  const int r1 = lane, ks = warp;
  for (int i = first1; i < n1; i += gridDim.x) {
    const Tile1 m = tile1(a, i);
    if (i != first1) issue1(m, routed_expert1(m));
    if (m.t != staged_t) {
      stage_bf16(xs, a.X + static_cast<size_t>(m.t) * K, K);
      __syncthreads();
      for (int kb = warp; kb < L.KB1; kb += kS1) {
        float v = xs[kb * 64 + lane] + xs[kb * 64 + 32 + lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) sxs[kb] = v;
      }
      __syncthreads();
      staged_t = m.t;
    }
    float acc_g = 0.0f, acc_u = 0.0f;
    bool ok = mbar_wait(&bars1[L.nbox1], par1, nullptr);
    for (int kb = ks; kb < L.KB1; kb += kS1) {
      const int b = kb / kBoxKB;
      ok &= mbar_wait(&bars1[b], par1, nullptr);
      const size_t boff = static_cast<size_t>(b) * box1;
      const float* xg = xs + kb * 64;
      acc_g += group_dot(qg + boff, r1, kb, xg, sxs[kb], sbg[kb * kR1 + r1]);
      acc_u += group_dot(qu + boff, r1, kb, xg, sxs[kb], sbu[kb * kR1 + r1]);
    }
    // every box of this use must have landed before its buffer is reused or the CTA exits
    for (int b = threadIdx.x; b <= L.nbox1; b += kThreads) ok &= mbar_wait(&bars1[b], par1, nullptr);
    if (!ok) record_status(a.status, MOE_ERR_TIMEOUT);
    red1[ks * kR1 + r1] = acc_g;
    red1[kS1 * kR1 + ks * kR1 + r1] = acc_u;
    __syncthreads();
    if (ks == 0) {
      float g = 0.0f, u = 0.0f;
#pragma unroll
      for (int s = 0; s < kS1; ++s) {
        g += red1[s * kR1 + r1];
        u += red1[kS1 * kR1 + s * kR1 + r1];
      }
      const float h = g / (1.0f + expf(-g)) * u;
      float* dst = m.shared ? a.h_shared + static_cast<size_t>(m.t) * a.I_shared
                            : a.h_routed + static_cast<size_t>(m.pair) * a.I;
      dst[m.n0 + r1] = h;
    }
    __syncthreads();
    par1 ^= 1;
  }

  grid_barrier(hdr, a.status);
  pdl_launch_dependents();

  // ---------------------------------------------------------------- phase 2: Y = sum_j w_j h_j Wd_j^T + shared
  uint32_t par2 = 0;
  const int r2 = threadIdx.x % kR2;
  const int slice = threadIdx.x / kR2;
  const int gpe = L.Imax / 64;
  const int P = k * L.KB2r + (has_shared ? L.KB2s : 0);
  for (int i = first2; i < n2; i += gridDim.x) {
    const int t = i / tiles2;
    const int n0 = (i % tiles2) * kR2;
    if (i != first2) {
      issue2(t, n0, false);
      issue2(t, n0, true);
    }
    // h of this token's routed experts (adjacent rows of h_routed) and of the shared expert
    stage_f32(hs, a.h_routed + static_cast<size_t>(t) * k * a.I, k * a.I);
    if (has_shared) stage_f32(hs + static_cast<size_t>(k) * a.I, a.h_shared + static_cast<size_t>(t) * a.I_shared,
                              a.I_shared);
    if (threadIdx.x < k) w2[threadIdx.x] = a.w[static_cast<size_t>(t) * k + threadIdx.x];
    if (threadIdx.x == 0 && has_shared) w2[k] = 1.0f;
    __syncthreads();
    for (int id = warp; id < L.nexp * gpe; id += kThreads / 32) {
      const int j = id / gpe, kb = id % gpe;
      const int Ij = (j == k) ? a.I_shared : a.I;
      if (kb * 64 >= Ij) continue;
      const float* x = hs + static_cast<size_t>(j) * a.I + kb * 64;
      float v = x[lane] + x[32 + lane];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) sx2[j * gpe + kb] = v;
    }
    __syncthreads();
    float acc = 0.0f;
    bool ok = true;
    for (int p = slice; p < P; p += kS2) {
      int j, kb;
      if (p < k * L.KB2r) {
        j = p / L.KB2r;
        kb = p % L.KB2r;
      } else {
        j = k;
        kb = p - k * L.KB2r;
      }
      ok &= mbar_wait(&bars2[j], par2, nullptr);
      const uint8_t* tile;
      uint32_t sbv;
      if (j < k) {
        tile = q2 + (static_cast<size_t>(j) * L.nbox2r + kb / kBoxKB) * box2;
        sbv = reinterpret_cast<const uint32_t*>(smem + L.sb2 + static_cast<size_t>(j) * L.sb2_slot)[kb * kR2 + r2];
      } else {
        tile = q2s + static_cast<size_t>(kb / kBoxKB) * box2;
        sbv = sb2s[kb * kR2 + r2];
      }
      const float dv = group_dot(tile, r2, kb, hs + static_cast<size_t>(j) * a.I + kb * 64, sx2[j * gpe + kb], sbv);
      acc = fmaf(w2[j], dv, acc);
    }
    for (int j = threadIdx.x; j < L.nexp; j += kThreads) ok &= mbar_wait(&bars2[j], par2, nullptr);
    if (!ok) record_status(a.status, MOE_ERR_TIMEOUT);
    red2[slice * kR2 + r2] = acc;
    __syncthreads();
    if (slice == 0) {
      float y = 0.0f;
#pragma unroll
      for (int s = 0; s < kS2; ++s) y += red2[s * kR2 + r2];
      a.Y[static_cast<size_t>(t) * a.d + n0 + r2] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
    }
    __syncthreads();
    par2 ^= 1;
  }
}

bool g_attr_set = false;

}  // namespace

size_t gemv_smem_bytes(int d, int I, int I_shared, int k) { return layout(d, I, I_shared, k).total; }

bool gemv_supported(int d, int I, int I_shared, int k) {
  const Layout L = layout(d, I, I_shared, k);
  return L.total <= 227 * 1024 && L.nbox1 + 1 <= 32 && L.nexp <= 32;
}

cudaError_t launch_gemv(const GemvArgs& a, const GemvMaps* routed, const GemvMaps* shared, void* ws,
                        cudaStream_t stream, bool pdl) {
  const Layout L = layout(a.d, a.I, a.I_shared, a.k);
  // TMA destinations: swizzled code boxes on 1024 bytes, group parameters on 128
  const bool aligned = L.q1 % 1024 == 0 && L.sb1 % 128 == 0 && L.sb1_slot % 128 == 0 && L.q2 % 1024 == 0 &&
                       L.q2s % 1024 == 0 && L.sb2 % 128 == 0 && L.sb2_slot % 128 == 0 && L.sb2s % 128 == 0 &&
                       L.bars % 8 == 0 && L.nbox1 + 1 <= 32 && L.nexp <= 32;
  if (!aligned) return cudaErrorInvalidValue;
  if (!g_attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    g_attr_set = true;
  }
  const GemvMaps* sh = shared ? shared : routed;  // unused when there is no shared expert
  const int n1 = a.T * a.k * (a.I / kR1) + (a.I_shared > 0 ? a.T * (a.I_shared / kR1) : 0);
  const int n2 = a.T * (a.d / kR2);
  int grid = n1 > n2 ? n1 : n2;
  if (grid > a.num_sms) grid = a.num_sms;

  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.total;
  timer_begin(kKGemvGateUp, stream);
  const cudaError_t err =
      cudaLaunchKernelEx(&cfg, decode_kernel, routed->q_gate, routed->q_up, routed->sb_gate, routed->sb_up,
                         routed->q_down, routed->sb_down, sh->q_gate, sh->q_up, sh->sb_gate, sh->sb_up, sh->q_down,
                         sh->sb_down, a, static_cast<WsHeader*>(ws));
  timer_end(kKGemvGateUp, stream);
  return err;
}

}  // namespace bm
