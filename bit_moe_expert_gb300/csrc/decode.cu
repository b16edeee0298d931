// Decode path (T <= 4 tokens): the expert projections as matrix-vector
// products on the CUDA cores.  "Perplexity's Lily Beats MLX-LM on MacBook M5",
// section "Prefill and decode are different problems": batch-1 decode is a
// GEMV bound by memory bandwidth that belongs on the vector ALUs; section
// "Decode: minimize bytes per token": the expert input projections are fused
// with the gate activation and the output projection with the routing scores
// and the shared expert.
//
// Design (sm_103a): one launch per layer, clusters of two CTAs, no grid-wide
// barrier.  A unit of work is one group of 64 intermediate features of one
// active expert (the shared expert's groups first, then the distinct routed
// experts of the call).  The two CTAs of a cluster split a unit:
//   gate/up  CTA r computes h = silu(x Wg^T) * (x Wu^T) for features
//            [64g + 32r, 64g + 32r + 32) of every token and writes them into
//            both CTAs' shared memory (distributed shared memory), then a
//            cluster barrier;
//   down     CTA r multiplies rows [r d/2, (r+1) d/2) of the down projection,
//            restricted to the group's 64 columns (one quantisation group, 32
//            bytes of codes per row), by the 64 h values and accumulates the
//            routing-weighted result in registers.
// Every byte of an active expert's three matrices is loaded once, by TMA,
// issued up front in few large boxes (the codes are stored group-major, so a
// group of many rows is one contiguous block); the next unit's loads start as
// soon as a buffer is free.
// Each cluster writes its partial output rows to global memory; the last 16
// CTAs to finish (an arrival counter) wait for the rest and sum the partials
// in a fixed order, so the result does not depend on timing.
//
// Arithmetic: a 4-bit code becomes the fp32 value 128 + q with one byte
// permute (exponent of 128, code in the low mantissa bits); products with x
// use packed fp32x2 FMAs; the affine map is applied once per 64-column group:
//   sum_k (q_k s + b) x_k = s * sum_k (128 + q_k) x_k + (b - 128 s) * sum_k x_k.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bm {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = kDecodeRowsGU;              // gate/up rows per CTA and unit (lane = row)
constexpr int kPairs = kThreads / 2;              // down rows are taken by thread pairs
constexpr int kMaxSlots = kMaxK * kGemvMaxT + 1;  // distinct experts of a call, plus the shared one
constexpr int kReducers = 16;
constexpr uint32_t kMagic128 = 0x43000000u;  // fp32 128.0: a code in bits 16..19 reads as 128 + q
constexpr long long kSpinLimitCycles = 4000000000ll;

__host__ __device__ constexpr int div_up(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  int KB1, half, nboxd, box_sr;
  size_t sb1_slot, qgu, qd, sbgu, sbd, accd, xs, sx, red, hb, wt, slot_e, misc, bars, total;
};

// TMA destinations start on 128 bytes.
__host__ __device__ inline Layout layout(int T, int d) {
  Layout L;
  L.KB1 = d / 64;
  L.half = d / 2;
  const int sr = d / 8;  // 128-byte super-rows (4 rows of 32 bytes) in a half of the down rows
  L.nboxd = div_up(sr, 256);
  L.box_sr = static_cast<int>(round_up(div_up(sr, L.nboxd), 8));
  L.sb1_slot = round_up(static_cast<size_t>(L.KB1) * kRows * 4, 128);
  size_t o = 0;
  L.qgu = o;  // gate codes [KB1][32 rows][32 B], then up codes
  o += 2ull * L.KB1 * kRows * 32;
  L.qd = o;  // down codes of the unit's group: [rows of this half][32 B]
  o += static_cast<size_t>(L.nboxd) * L.box_sr * 128;
  L.sbgu = o;
  o += 2 * L.sb1_slot;
  L.sbd = o;
  o += static_cast<size_t>(L.nboxd) * L.box_sr * 16;
  L.accd = o;  // down accumulators [rows of this half][T]
  o += static_cast<size_t>(L.half) * T * 4;
  o = round_up(o, 16);
  L.xs = o;  // x of every token, fp32 [T][d]
  o += static_cast<size_t>(T) * d * 4;
  L.sx = o;  // per-group sums of x [T][d/64]
  o += static_cast<size_t>(T) * L.KB1 * 4;
  o = round_up(o, 16);
  L.red = o;  // gate and up partial dots [2][warp][row][T]
  o += 2ull * kWarps * kRows * T * 4;
  L.hb = o;  // h of the unit's 64 features, two buffers [2][T][64]
  o += 2ull * T * 64 * 4;
  L.wt = o;  // routing weight of each slot for each token [slot][T]
  o += static_cast<size_t>(kMaxSlots) * T * 4;
  L.slot_e = o;  // expert of each slot
  o += kMaxSlots * 4;
  L.misc = o;  // slot count, arrival ticket
  o += 16;
  o = round_up(o, 8);
  L.bars = o;  // gate/up, then nboxd down boxes
  o += static_cast<size_t>(1 + L.nboxd) * 8;
  L.total = o + 128;  // room to align the dynamic shared memory base
  return L;
}

struct Unit {
  int g, slot;
  bool shared;
};

// The shared expert's groups come first (they need no routing), then each
// routed slot's groups.
__device__ __forceinline__ Unit unit_of(int u, int Gs, int G, bool has_shared) {
  Unit m;
  if (u < Gs) {
    m.shared = true;
    m.g = u;
    m.slot = 0;
  } else {
    const int v = u - Gs;
    m.shared = false;
    m.slot = (has_shared ? 1 : 0) + v / G;
    m.g = v % G;
  }
  return m;
}

// Four fp32 pairs (128 + q) for the eight codes of one word, in k order.
__device__ __forceinline__ void codes8(uint32_t w, float2 (&q)[4]) {
  const uint32_t lo = w & 0x0F0F0F0Fu;         // codes 0, 2, 4, 6 in bytes 0..3
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // codes 1, 3, 5, 7
  q[0] = make_float2(__uint_as_float(prmt(lo, kMagic128, 0x7054)), __uint_as_float(prmt(hi, kMagic128, 0x7054)));
  q[1] = make_float2(__uint_as_float(prmt(lo, kMagic128, 0x7154)), __uint_as_float(prmt(hi, kMagic128, 0x7154)));
  q[2] = make_float2(__uint_as_float(prmt(lo, kMagic128, 0x7254)), __uint_as_float(prmt(hi, kMagic128, 0x7254)));
  q[3] = make_float2(__uint_as_float(prmt(lo, kMagic128, 0x7354)), __uint_as_float(prmt(hi, kMagic128, 0x7354)));
}

// sum over eight codes of (128 + q) * x for every token; x at xp[t * stride].
template <int kT>
__device__ __forceinline__ void word_dot(uint32_t w, const float* xp, int stride, float2 (&acc)[kT]) {
  float2 q[4];
  codes8(w, q);
#pragma unroll
  for (int t = 0; t < kT; ++t) {
    const float4 xa = *reinterpret_cast<const float4*>(xp + t * stride);
    const float4 xb = *reinterpret_cast<const float4*>(xp + t * stride + 4);
    acc[t] = f32x2_fma(q[0], make_float2(xa.x, xa.y), acc[t]);
    acc[t] = f32x2_fma(q[1], make_float2(xa.z, xa.w), acc[t]);
    acc[t] = f32x2_fma(q[2], make_float2(xb.x, xb.y), acc[t]);
    acc[t] = f32x2_fma(q[3], make_float2(xb.z, xb.w), acc[t]);
  }
}

// One gate/up row's contribution from one 64-column group, for every token.
//   codes: [KB][32 rows][32 bytes]; xs: x of every token [T][d]; sx: group sums [T][KB]
template <int kT>
__device__ __forceinline__ void group_dot(const uint8_t* codes, int row, int kb, const float* xs, int d,
                                          const float* sx, int KB, uint32_t sbv, float (&out)[kT]) {
  const uint8_t* rp = codes + (kb * kRows + row) * 32;
  const uint4 wa = *reinterpret_cast<const uint4*>(rp);
  const uint4 wb = *reinterpret_cast<const uint4*>(rp + 16);
  float2 a0[kT], a1[kT];
#pragma unroll
  for (int t = 0; t < kT; ++t) a0[t] = a1[t] = make_float2(0.0f, 0.0f);
  const float* xg = xs + kb * 64;
  word_dot<kT>(wa.x, xg + 0, d, a0);
  word_dot<kT>(wa.y, xg + 8, d, a1);
  word_dot<kT>(wa.z, xg + 16, d, a0);
  word_dot<kT>(wa.w, xg + 24, d, a1);
  word_dot<kT>(wb.x, xg + 32, d, a0);
  word_dot<kT>(wb.y, xg + 40, d, a1);
  word_dot<kT>(wb.z, xg + 48, d, a0);
  word_dot<kT>(wb.w, xg + 56, d, a1);
  const float s = __uint_as_float(sbv << 16);
  const float b = __uint_as_float(sbv & 0xFFFF0000u);
  const float c = b - 128.0f * s;
#pragma unroll
  for (int t = 0; t < kT; ++t) {
    const float p = (a0[t].x + a0[t].y) + (a1[t].x + a1[t].y);
    out[t] += fmaf(s, p, c * sx[t * KB + kb]);
  }
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

template <int kT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap qg_r, const __grid_constant__ CUtensorMap qu_r,
                  const __grid_constant__ CUtensorMap sbg_r, const __grid_constant__ CUtensorMap sbu_r,
                  const __grid_constant__ CUtensorMap qd_r, const __grid_constant__ CUtensorMap sbd_r,
                  const __grid_constant__ CUtensorMap qg_s, const __grid_constant__ CUtensorMap qu_s,
                  const __grid_constant__ CUtensorMap sbg_s, const __grid_constant__ CUtensorMap sbu_s,
                  const __grid_constant__ CUtensorMap qd_s, const __grid_constant__ CUtensorMap sbd_s,
                  DecodeArgs a, WsHeader* hdr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int d = a.d;
  const Layout L = layout(kT, d);
  const bool has_shared = a.I_shared > 0;
  const int G = a.I / 64, Gs = a.I_shared / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);

  uint8_t* qg = smem + L.qgu;
  uint8_t* qu = qg + static_cast<size_t>(L.KB1) * kRows * 32;
  const uint8_t* qd = smem + L.qd;
  const uint32_t* sbg = reinterpret_cast<const uint32_t*>(smem + L.sbgu);
  const uint32_t* sbu = reinterpret_cast<const uint32_t*>(smem + L.sbgu + L.sb1_slot);
  const uint32_t* sbd = reinterpret_cast<const uint32_t*>(smem + L.sbd);
  float* accd = reinterpret_cast<float*>(smem + L.accd);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* sx = reinterpret_cast<float*>(smem + L.sx);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* hb = reinterpret_cast<float*>(smem + L.hb);
  float* wt = reinterpret_cast<float*>(smem + L.wt);
  int* slot_e = reinterpret_cast<int*>(smem + L.slot_e);
  int* misc = reinterpret_cast<int*>(smem + L.misc);
  uint64_t* bar_gu = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* bar_d = bar_gu + 1;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 1 + L.nboxd; ++b) mbar_init(&bar_gu[b], 1);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < L.half * kT; i += kThreads) accd[i] = 0.0f;
  for (int i = threadIdx.x; i < kMaxSlots * kT; i += kThreads) wt[i] = 0.0f;
  __syncthreads();
  cluster_arrive_relaxed();  // matched by a wait before the first write into the other CTA

  // One lane of warp 0 issues every load of a unit: gate and up codes (one box
  // each: 32 rows x every group), their group parameters, and the down rows of
  // this CTA's half for the unit's group (codes and parameters, nboxd boxes).
  auto issue = [&](const Unit& m, int e) {
    const int n0 = m.g * 64 + static_cast<int>(rank) * kRows;
    mbar_arrive_expect_tx(&bar_gu[0], static_cast<uint32_t>(2 * L.KB1 * kRows * (32 + 4)));
    tma_load_3d(qg, m.shared ? &qg_s : &qg_r, &bar_gu[0], 0, n0, e * L.KB1);
    tma_load_3d(qu, m.shared ? &qu_s : &qu_r, &bar_gu[0], 0, n0, e * L.KB1);
    tma_load_3d(smem + L.sbgu, m.shared ? &sbg_s : &sbg_r, &bar_gu[0], n0, 0, e);
    tma_load_3d(smem + L.sbgu + L.sb1_slot, m.shared ? &sbu_s : &sbu_r, &bar_gu[0], n0, 0, e);
    const int Ge = m.shared ? Gs : G;
    for (int b = 0; b < L.nboxd; ++b) {
      const int sr0 = static_cast<int>(rank) * (L.half / 4) + b * L.box_sr;
      mbar_arrive_expect_tx(&bar_d[b], static_cast<uint32_t>(L.box_sr * (128 + 16)));
      tma_load_3d(smem + L.qd + static_cast<size_t>(b) * L.box_sr * 128, m.shared ? &qd_s : &qd_r, &bar_d[b], 0,
                  sr0, e * Ge + m.g);
      tma_load_3d(smem + L.sbd + static_cast<size_t>(b) * L.box_sr * 16, m.shared ? &sbd_s : &sbd_r, &bar_d[b], 0,
                  sr0, e * Ge + m.g);
    }
  };

  const int u0 = cl;
  const int rs0 = has_shared ? 1 : 0;
  // Shared-expert weights do not depend on the previous kernels: start them first.
  if (u0 < Gs && threadIdx.x == 0) issue(unit_of(u0, Gs, G, has_shared), 0);
  pdl_wait();  // routing, X and the previous layer's use of the workspace

  if (warp == 0) {
    // Distinct experts of the call in order of first appearance, and the
    // routing weight of each for each token.
    const int na = kT * a.k;
    int nsl = rs0;
    if (na <= 32) {
      // one assignment per lane: a lane whose expert no lower lane holds opens a slot
      const bool valid = lane < na;
      int e = valid ? __ldg(a.ids + lane) : -1 - lane;
      const float wi = valid ? __ldg(a.w + lane) : 0.0f;
      if (valid && (e < 0 || e >= a.E)) {
        record_status(a.status, MOE_ERR_INVALID_ARG);
        e = 0;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int leader = __ffs(peers) - 1;
      const unsigned opens = __ballot_sync(0xffffffffu, valid && leader == lane);
      const int my_slot = rs0 + __popc(opens & ((1u << lane) - 1u));
      const int slot = __shfl_sync(0xffffffffu, my_slot, leader);
      if (valid) {
        if (leader == lane) slot_e[slot] = e;
        wt[slot * kT + lane / a.k] = wi;
      }
      nsl = rs0 + __popc(opens);
    } else {
      // more assignments than lanes: walk them in order
      for (int i = 0; i < na; ++i) {
        int e = __ldg(a.ids + i);
        const float wi = __ldg(a.w + i);
        if (e < 0 || e >= a.E) {
          if (lane == 0) record_status(a.status, MOE_ERR_INVALID_ARG);
          e = 0;
        }
        int slot = -1;
        for (int c0 = rs0; c0 < nsl && slot < 0; c0 += 32) {
          const unsigned hit = __ballot_sync(0xffffffffu, c0 + lane < nsl && slot_e[c0 + lane] == e);
          if (hit) slot = c0 + __ffs(hit) - 1;
        }
        if (slot < 0) slot = nsl++;
        __syncwarp();
        if (lane == 0) {
          slot_e[slot] = e;
          wt[slot * kT + i / a.k] = wi;
        }
        __syncwarp();
      }
    }
    __syncwarp();
    if (lane == 0) {
      misc[0] = nsl - rs0;
      if (has_shared) {
        slot_e[0] = 0;
        for (int t = 0; t < kT; ++t) wt[t] = 1.0f;
      }
    }
    __syncwarp();
    // the routed unit's loads start as soon as its expert is known
    const int U = Gs + (nsl - rs0) * G;
    if (lane == 0 && u0 >= Gs && u0 < U) {
      const Unit m = unit_of(u0, Gs, G, has_shared);
      issue(m, slot_e[m.slot]);
    }
  } else {
    // the other warps stage x (bf16 -> fp32) and its per-group sums
    const int n8 = kT * d / 8;
    for (int f = threadIdx.x - 32; f < n8; f += kThreads - 32) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.X) + f);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float4* d4 = reinterpret_cast<float4*>(xs + f * 8);
      d4[0] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                          __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
      d4[1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                          __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kThreads - 32) : "memory");  // warps 1..15 only
    for (int idx = warp - 1; idx < kT * L.KB1; idx += kWarps - 1) {
      const float* xg = xs + (idx / L.KB1) * d + (idx % L.KB1) * 64;
      float v = xg[lane] + xg[32 + lane];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) sx[idx] = v;
    }
  }
  __syncthreads();
  const int U = Gs + misc[0] * G;
  pdl_launch_dependents();

  const int p = threadIdx.x >> 1;  // down rows p, p + 256, ... of this CTA's half
  const int hf = threadIdx.x & 1;  // which 32 of the group's 64 columns
  uint32_t par = 0;
  int buf = 0;
  bool waited = false;
  bool ok = true;
  for (int u = u0; u < U; u += ncl) {
    const Unit m = unit_of(u, Gs, G, has_shared);
    // ---------------------------------------------------- gate/up: lane = row, warp = K slice
    float ag[kT], au[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) ag[t] = au[t] = 0.0f;
    ok &= mbar_wait(&bar_gu[0], par, nullptr);
    for (int kb = warp; kb < L.KB1; kb += kWarps) {
      group_dot<kT>(qg, lane, kb, xs, d, sx, L.KB1, sbg[kb * kRows + lane], ag);
      group_dot<kT>(qu, lane, kb, xs, d, sx, L.KB1, sbu[kb * kRows + lane], au);
    }
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      red[(warp * kRows + lane) * kT + t] = ag[t];
      red[((kWarps + warp) * kRows + lane) * kT + t] = au[t];
    }
    if (!waited) {
      cluster_wait();  // the other CTA of the cluster is running
      waited = true;
    }
    __syncthreads();
    float* hbb = hb + buf * kT * 64;
    if (warp < kT) {
      // token t = warp: h of this CTA's 32 features, into both CTAs
      const int t = warp;
      float g = 0.0f, uu = 0.0f;
#pragma unroll
      for (int s = 0; s < kWarps; ++s) {
        g += red[(s * kRows + lane) * kT + t];
        uu += red[((kWarps + s) * kRows + lane) * kT + t];
      }
      const float h = g / (1.0f + expf(-g)) * uu;
      float* dst = hbb + t * 64 + static_cast<int>(rank) * kRows + lane;
      *dst = h;
      st_cluster_f32(mapa_shared(smem_u32(dst), rank ^ 1u), h);
    }
    cluster_sync();  // all 64 h values of the group are in both CTAs
    // ---------------------------------------------------- down: thread pair = row, 32 columns each
    float wts[kT], hs[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      wts[t] = wt[m.slot * kT + t];
      const float* hv = hbb + t * 64;
      float v = 0.0f;
#pragma unroll 8
      for (int i = 0; i < 64; ++i) v += hv[i];  // broadcast reads; every thread gets the same sum
      hs[t] = v;
    }
    for (int b = 0; b < L.nboxd; ++b) ok &= mbar_wait(&bar_d[b], par, nullptr);
    for (int row = p; row < L.half; row += kPairs) {
      float2 pp[kT];
#pragma unroll
      for (int t = 0; t < kT; ++t) pp[t] = make_float2(0.0f, 0.0f);
      const uint4 w = *reinterpret_cast<const uint4*>(qd + row * 32 + hf * 16);
      const float* hp = hbb + hf * 32;
      word_dot<kT>(w.x, hp + 0, 64, pp);
      word_dot<kT>(w.y, hp + 8, 64, pp);
      word_dot<kT>(w.z, hp + 16, 64, pp);
      word_dot<kT>(w.w, hp + 24, 64, pp);
      const uint32_t sbv = sbd[row];
      const float s = __uint_as_float(sbv << 16);
      const float c = __uint_as_float(sbv & 0xFFFF0000u) - 128.0f * s;
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        float pv = pp[t].x + pp[t].y;
        pv += __shfl_xor_sync(0xffffffffu, pv, 1);
        const float y = fmaf(s, pv, c * hs[t]);
        if (hf == 0 && wts[t] != 0.0f) accd[row * kT + t] = fmaf(wts[t], y, accd[row * kT + t]);
      }
    }
    __syncthreads();  // every box of this unit has been read
    if (u + ncl < U && threadIdx.x == 0) {
      const Unit nx = unit_of(u + ncl, Gs, G, has_shared);
      issue(nx, nx.shared ? 0 : slot_e[nx.slot]);
    }
    par ^= 1;
    buf ^= 1;
  }
  if (!waited) cluster_wait();
  if (!ok) record_status(a.status, MOE_ERR_TIMEOUT);

  // ---------------------------------------------------- this cluster's partial output rows
  float* part = a.part + static_cast<size_t>(cl) * kT * d + static_cast<int>(rank) * L.half;
  for (int i = threadIdx.x; i < L.half * kT; i += kThreads) {
    const int t = i / L.half, row = i % L.half;
    part[static_cast<size_t>(t) * d + row] = accd[row * kT + t];
  }
  __syncthreads();
  if (threadIdx.x == 0) misc[1] = static_cast<int>(atom_add_acq_rel_gpu(&hdr->dec_arrive, 1u));
  __syncthreads();
  const int R = min(kReducers, static_cast<int>(gridDim.x));
  const int ticket = misc[1];
  if (ticket < static_cast<int>(gridDim.x) - R) return;

  // ---------------------------------------------------- the last R CTAs: Y = sum of the partials
  const int slice = ticket - (static_cast<int>(gridDim.x) - R);
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    while (ld_acquire_gpu(&hdr->dec_arrive) < gridDim.x) {
      if (clock64() - t0 > kSpinLimitCycles) {
        record_status(a.status, MOE_ERR_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  const int d4 = d / 4;
  const int per = div_up(d4, R);
  const int f0 = slice * per, f1 = min(d4, f0 + per);  // float4 columns of this reducer
  // warp w sums the partials of clusters w, w + 16, ...; then the 16 sums are
  // added in warp order: a fixed order, whatever the timing
  float4* red4 = reinterpret_cast<float4*>(smem + L.qgu);
  const size_t red4_cap = (2ull * L.KB1 * kRows * 32) / (kWarps * kT * 16);  // float4 per warp and token
  const int cw = red4_cap < 32 ? static_cast<int>(red4_cap) : 32;
  for (int j0 = f0; j0 < f1; j0 += cw) {
    const int j = j0 + lane;
    if (lane < cw) {
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        float4 sacc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (j < f1) {
          for (int c = warp; c < ncl; c += kWarps) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part + (static_cast<size_t>(c) * kT + t) * d) + j);
            sacc.x += v.x;
            sacc.y += v.y;
            sacc.z += v.z;
            sacc.w += v.w;
          }
        }
        red4[(warp * kT + t) * cw + lane] = sacc;
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kT * cw; i += kThreads) {
      const int t = i / cw, jj = j0 + i % cw;
      if (jj < f1) {
        float4 y = red4[t * cw + i % cw];
        for (int w = 1; w < kWarps; ++w) {
          const float4 v = red4[(w * kT + t) * cw + i % cw];
          y.x += v.x;
          y.y += v.y;
          y.z += v.z;
          y.w += v.w;
        }
        const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(y.x))) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(y.y))) << 16);
        const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(y.z))) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(y.w))) << 16);
        *reinterpret_cast<uint2*>(a.Y + static_cast<size_t>(t) * d + jj * 4) = make_uint2(lo, hi);
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (atom_add_acq_rel_gpu(&hdr->dec_done, 1u) == static_cast<uint32_t>(R - 1)) {
      // every CTA has arrived and every reducer has read the counter: reset for the next call
      hdr->dec_arrive = 0;
      hdr->dec_done = 0;
      __threadfence();
    }
  }
}

template <int kT>
cudaError_t launch_t(const DecodeArgs& a, const DecodeMaps* routed, const DecodeMaps* sh, WsHeader* hdr, int grid,
                     size_t smem, cudaStream_t stream, bool pdl) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<kT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  return cudaLaunchKernelEx(&cfg, decode_kernel<kT>, routed->q_gate, routed->q_up, routed->sb_gate, routed->sb_up,
                            routed->q_down, routed->sb_down, sh->q_gate, sh->q_up, sh->sb_gate, sh->sb_up,
                            sh->q_down, sh->sb_down, a, hdr);
}

}  // namespace

bool decode_supported(int T, int d, int I, int I_shared, int k) {
  if (T < 1 || T > kGemvMaxT || k > kMaxK) return false;
  const Layout L = layout(T, d);
  return L.total <= 227 * 1024 && L.KB1 <= 256 && L.nboxd <= 8 && d % 64 == 0 && I % 64 == 0 &&
         I_shared % 64 == 0;
}

size_t decode_partial_bytes(int T, int d) { return static_cast<size_t>(kDecodeMaxClusters) * T * d * 4; }

int decode_box_superrows(int d) { return layout(1, d).box_sr; }

cudaError_t launch_decode(const DecodeArgs& a, const DecodeMaps* routed, const DecodeMaps* shared, void* ws,
                          cudaStream_t stream, bool pdl) {
  const Layout L = layout(a.T, a.d);
  const bool aligned = L.qgu % 128 == 0 && L.qd % 128 == 0 && L.sbgu % 128 == 0 && L.sb1_slot % 128 == 0 &&
                       L.sbd % 128 == 0 && (L.box_sr * 16) % 128 == 0 && L.bars % 8 == 0;
  if (!aligned || !decode_supported(a.T, a.d, a.I, a.I_shared, a.k)) return cudaErrorInvalidValue;
  const DecodeMaps* sh = shared ? shared : routed;  // never read without a shared expert
  const int distinct = a.T * a.k < a.E ? a.T * a.k : a.E;
  const int units = a.I_shared / 64 + distinct * (a.I / 64);
  int ncl = a.num_sms / 2;
  if (ncl > units) ncl = units;
  if (ncl > kDecodeMaxClusters) ncl = kDecodeMaxClusters;
  if (ncl < 1) ncl = 1;
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  timer_begin(kKDecode, stream);
  cudaError_t err;
  switch (a.T) {
    case 1: err = launch_t<1>(a, routed, sh, hdr, 2 * ncl, L.total, stream, pdl); break;
    case 2: err = launch_t<2>(a, routed, sh, hdr, 2 * ncl, L.total, stream, pdl); break;
    case 3: err = launch_t<3>(a, routed, sh, hdr, 2 * ncl, L.total, stream, pdl); break;
    default: err = launch_t<4>(a, routed, sh, hdr, 2 * ncl, L.total, stream, pdl); break;
  }
  timer_end(kKDecode, stream);
  return err;
}

}  // namespace bm
