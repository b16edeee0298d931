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
// Each cluster writes its partial output rows; after one barrier over the
// grid every CTA sums a few output rows over the clusters in a fixed order, so
// the result does not depend on timing.
//
// Arithmetic: a 4-bit code becomes the fp32 value 128 + q with one byte
// permute (exponent of 128, code in the low mantissa bits); products with x
// use packed fp32x2 FMAs; the affine map is applied once per 64-column group:
//   sum_k (q_k s + b) x_k = s * sum_k (128 + q_k) x_k + (b - 128 s) * sum_k x_k.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace bm {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = kDecodeRowsGU;              // gate/up rows per CTA and unit (lane = row)
constexpr int kPairs = kThreads / 2;              // down rows are taken by thread pairs
constexpr int kChunkGroups = kDecodeChunkGroups;  // gate/up codes arrive in chunks of groups, one barrier each
constexpr int kMaxSlots = kMaxK * kGemvMaxT + 1;  // distinct experts of a call, plus the shared one
constexpr uint32_t kMagic128 = 0x43000000u;  // fp32 128.0: a code in bits 16..19 reads as 128 + q

__host__ __device__ constexpr int div_up(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  int KB1, nchunk, half, nboxd, box_sr;
  size_t sb1_slot, qgu, qd, sbgu, sbd, accd, xs, sx, red, hb, hsb, wt, slot_e, rid, misc, bars, total;
};

// TMA destinations start on 128 bytes.
__host__ __device__ inline Layout layout(int T, int d) {
  Layout L;
  L.KB1 = d / 64;
  L.nchunk = div_up(L.KB1, kChunkGroups);
  L.half = d / 2;
  const int sr = d / 8;  // 128-byte super-rows (4 rows of 32 bytes) in a half of the down rows
  L.nboxd = div_up(sr, 256);
  L.box_sr = static_cast<int>(round_up(div_up(sr, L.nboxd), 8));
  L.sb1_slot = round_up(static_cast<size_t>(L.KB1) * kRows * 4, 128);
  size_t o = 0;
  L.qgu = o;  // gate codes [KB1][32 rows][32 B], then up codes
  o += 2ull * L.nchunk * kChunkGroups * kRows * 32;
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
  L.sx = o;  // sums of x over each half group of 32 columns [T][d/32]
  o += static_cast<size_t>(T) * 2 * L.KB1 * 4;
  o = round_up(o, 16);
  L.red = o;  // gate and up partial dots [2][warp][row][T]
  o += 2ull * kWarps * kRows * T * 4;
  L.hb = o;  // h of the unit's 64 features, two buffers [2][T][64]
  o += 2ull * T * 64 * 4;
  L.hsb = o;  // the two halves' sums of h, [2][T][2]
  o += 2ull * T * 2 * 4;
  L.wt = o;  // routing weight of each slot for each token [slot][T]
  o += static_cast<size_t>(kMaxSlots) * T * 4;
  L.slot_e = o;  // expert of each slot
  o += kMaxSlots * 4;
  L.rid = o;  // the call's assignments: expert [T*k], weight [T*k], slot [T*k]
  o += 3ull * T * kMaxK * 4;
  L.misc = o;  // slot count, arrival ticket
  o += 16;
  o = round_up(o, 8);
  L.bars = o;  // gate/up code chunks, gate/up group parameters, down boxes, two h exchanges
  o += static_cast<size_t>(L.nchunk + 1 + L.nboxd + 2) * 8;
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

// One gate/up row's contribution from half (32 columns) of one group, for
// every token, for gate and up together (they share the x loads).
//   qg, qu: codes [groups][32 rows][32 bytes]; xs: x [T][d]; sx: sums of x
//   over each half group [T][nh]
template <int kT>
__device__ __forceinline__ void half_group_dot2(const uint8_t* qg, const uint8_t* qu, int row, int kb, int hh,
                                                const float* xs, int d, const float* sx, int nh, uint32_t sbg,
                                                uint32_t sbu, float (&og)[kT], float (&ou)[kT]) {
  const int off = (kb * kRows + row) * 32 + hh * 16;
  const uint4 wg = *reinterpret_cast<const uint4*>(qg + off);
  const uint4 wu = *reinterpret_cast<const uint4*>(qu + off);
  const uint32_t gw[4] = {wg.x, wg.y, wg.z, wg.w};
  const uint32_t uw[4] = {wu.x, wu.y, wu.z, wu.w};
  float2 ag[kT], au[kT];
#pragma unroll
  for (int t = 0; t < kT; ++t) ag[t] = au[t] = make_float2(0.0f, 0.0f);
  const float* xg = xs + kb * 64 + hh * 32;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float2 qa[4], qb[4];
    codes8(gw[j], qa);
    codes8(uw[j], qb);
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      const float4 xa = *reinterpret_cast<const float4*>(xg + t * d + 8 * j);
      const float4 xb = *reinterpret_cast<const float4*>(xg + t * d + 8 * j + 4);
      ag[t] = f32x2_fma(qa[0], make_float2(xa.x, xa.y), ag[t]);
      au[t] = f32x2_fma(qb[0], make_float2(xa.x, xa.y), au[t]);
      ag[t] = f32x2_fma(qa[1], make_float2(xa.z, xa.w), ag[t]);
      au[t] = f32x2_fma(qb[1], make_float2(xa.z, xa.w), au[t]);
      ag[t] = f32x2_fma(qa[2], make_float2(xb.x, xb.y), ag[t]);
      au[t] = f32x2_fma(qb[2], make_float2(xb.x, xb.y), au[t]);
      ag[t] = f32x2_fma(qa[3], make_float2(xb.z, xb.w), ag[t]);
      au[t] = f32x2_fma(qb[3], make_float2(xb.z, xb.w), au[t]);
    }
  }
  const float s1 = __uint_as_float(sbg << 16), c1 = __uint_as_float(sbg & 0xFFFF0000u) - 128.0f * s1;
  const float s2 = __uint_as_float(sbu << 16), c2 = __uint_as_float(sbu & 0xFFFF0000u) - 128.0f * s2;
#pragma unroll
  for (int t = 0; t < kT; ++t) {
    const float sxv = sx[t * nh + 2 * kb + hh];
    og[t] += fmaf(s1, ag[t].x + ag[t].y, c1 * sxv);
    ou[t] += fmaf(s2, au[t].x + au[t].y, c2 * sxv);
  }
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

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
  const bool fused = a.logits != nullptr;
  // with fused routing the last cluster takes no unit: its first CTA writes the routing outputs
  const int ncl = static_cast<int>(gridDim.x >> 1) - (fused ? 1 : 0);
  const bool bookkeeper = fused && cl == ncl && rank == 0;

  uint8_t* qg = smem + L.qgu;
  uint8_t* qu = qg + static_cast<size_t>(L.nchunk) * kChunkGroups * kRows * 32;
  const uint8_t* qd = smem + L.qd;
  const uint32_t* sbg = reinterpret_cast<const uint32_t*>(smem + L.sbgu);
  const uint32_t* sbu = reinterpret_cast<const uint32_t*>(smem + L.sbgu + L.sb1_slot);
  const uint32_t* sbd = reinterpret_cast<const uint32_t*>(smem + L.sbd);
  float* accd = reinterpret_cast<float*>(smem + L.accd);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* sx = reinterpret_cast<float*>(smem + L.sx);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* hb = reinterpret_cast<float*>(smem + L.hb);
  float* hsb = reinterpret_cast<float*>(smem + L.hsb);
  float* wt = reinterpret_cast<float*>(smem + L.wt);
  int* slot_e = reinterpret_cast<int*>(smem + L.slot_e);
  int* s_ids = reinterpret_cast<int*>(smem + L.rid);
  float* s_w = reinterpret_cast<float*>(smem + L.rid + static_cast<size_t>(kT) * kMaxK * 4);
  int* s_slot = reinterpret_cast<int*>(smem + L.rid + 2ull * kT * kMaxK * 4);
  int* misc = reinterpret_cast<int*>(smem + L.misc);
  uint64_t* bar_gu = reinterpret_cast<uint64_t*>(smem + L.bars);  // one per code chunk
  uint64_t* bar_sb = bar_gu + L.nchunk;
  uint64_t* bar_d = bar_sb + 1;
  uint64_t* bar_h = bar_d + L.nboxd;  // [2]: the other CTA's h values of a unit have arrived

  if (threadIdx.x == 0) {
    for (int b = 0; b < L.nchunk + 1 + L.nboxd; ++b) mbar_init(&bar_gu[b], 1);
    // an h exchange completes with the expected bytes from the other CTA, one
    // arrival with the byte count and one per exchanging warp of this CTA
    mbar_init(&bar_h[0], 1 + kT);
    mbar_init(&bar_h[1], 1 + kT);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < L.half * kT; i += kThreads) accd[i] = 0.0f;
  for (int i = threadIdx.x; i < kMaxSlots * kT; i += kThreads) wt[i] = 0.0f;
  __syncthreads();
  cluster_arrive_relaxed();  // matched by a wait before the first write into the other CTA

  // The lanes of warp 0 issue a unit's loads in parallel: lane c < nchunk the
  // gate and up codes of groups [8c, 8c+8) (32 rows each), lane nchunk the
  // gate/up group parameters, the next nboxd lanes the down rows of this CTA's
  // half for the unit's group (codes and parameters).
  // Warp 0 issues a unit's loads without divergence: first every barrier's
  // byte count (one lane per barrier), then one TMA copy per lane:
  //   copies 0, 1:               gate and up group parameters
  //   copies 2c+2, 2c+3:         gate and up codes of groups [8c, 8c+8), 32 rows (c < nchunk)
  //   then per down box b:       down codes and parameters of this CTA's half, the unit's group
  auto issue = [&](const Unit& m, int e) {
    const uint64_t pol = l2_policy_evict_first();  // every weight byte is read once
    const int n0 = m.g * 64 + static_cast<int>(rank) * kRows;
    const int Ge = m.shared ? Gs : G;
    const uint32_t cbytes = kChunkGroups * kRows * 32;
    if (lane < L.nchunk + 1 + L.nboxd) {
      uint64_t* bar;
      uint32_t bytes;
      if (lane < L.nchunk) {
        bar = &bar_gu[lane];
        bytes = 2 * cbytes;
      } else if (lane == L.nchunk) {
        bar = bar_sb;
        bytes = static_cast<uint32_t>(2 * L.KB1 * kRows * 4);
      } else {
        bar = &bar_d[lane - L.nchunk - 1];
        bytes = static_cast<uint32_t>(L.box_sr * (128 + 16));
      }
      mbar_arrive_expect_tx(bar, bytes);
    }
    __syncwarp();
    const int ncopy = 2 * (L.nchunk + 1 + L.nboxd);
    if (lane < ncopy) {
      // the group parameters first: every gate/up product needs them
      const int slot = lane >> 1, second = lane & 1;
      const int which = slot == 0 ? L.nchunk : slot - 1 < L.nchunk ? slot - 1 : slot;
      const CUtensorMap* map;
      void* dst;
      uint64_t* bar;
      int c1, c2;
      if (which < L.nchunk) {
        map = second ? (m.shared ? &qu_s : &qu_r) : (m.shared ? &qg_s : &qg_r);
        dst = (second ? qu : qg) + static_cast<size_t>(which) * cbytes;
        bar = &bar_gu[which];
        c1 = n0;
        c2 = e * L.KB1 + which * kChunkGroups;
      } else if (which == L.nchunk) {
        map = second ? (m.shared ? &sbu_s : &sbu_r) : (m.shared ? &sbg_s : &sbg_r);
        dst = smem + L.sbgu + (second ? L.sb1_slot : 0);
        bar = bar_sb;
        c1 = 0;
        c2 = e;
      } else {
        const int b = which - L.nchunk - 1;
        map = second ? (m.shared ? &sbd_s : &sbd_r) : (m.shared ? &qd_s : &qd_r);
        dst = second ? smem + L.sbd + static_cast<size_t>(b) * L.box_sr * 16
                     : smem + L.qd + static_cast<size_t>(b) * L.box_sr * 128;
        bar = &bar_d[b];
        c1 = static_cast<int>(rank) * (L.half / 4) + b * L.box_sr;
        c2 = e * Ge + m.g;
      }
      // the gate/up parameter boxes start at row n0 (their first coordinate)
      tma_load_3d_hint(dst, map, bar, which == L.nchunk ? n0 : 0, c1, c2, pol);
    }
  };

  const int u0 = cl < ncl ? cl : 0x3FFFFFFF;  // the routing cluster has no unit
  const int rs0 = has_shared ? 1 : 0;
  // Shared-expert weights do not depend on the previous kernels: start them
  // first.  Tensor maps, router logits and X are only pulled towards the SM
  // (the logits and X are read after the wait; an L2 prefetch of a line the
  // previous kernel still writes is harmless: L2 is where writes land).
  if (warp == 0 && u0 < Gs) issue(unit_of(u0, Gs, G, has_shared), 0);
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&qg_r);
    tma_prefetch_desc(&qu_r);
    tma_prefetch_desc(&sbg_r);
    tma_prefetch_desc(&sbu_r);
    tma_prefetch_desc(&qd_r);
    tma_prefetch_desc(&sbd_r);
  }
  if (warp == 1) {
    const char* lg = reinterpret_cast<const char*>(a.logits);
    const char* xp = reinterpret_cast<const char*>(a.X);
    if (lg)
      for (int off = lane * 128; off < kT * a.E * 4; off += 32 * 128) prefetch_l2(lg + off);
    for (int off = lane * 128; off < kT * d * 2; off += 32 * 128) prefetch_l2(xp + off);
  }
  pdl_wait();  // routing, X and the previous layer's use of the workspace

  const int na = kT * a.k;
  float sel_v = 0.0f;  // fused routing: this lane's selected logit (warps < kT)
  if (warp < kT) {
    // the call's assignments: routed here (one warp per token) or read from memory
    if (fused) {
      // the selection now; its weights after the expert loads have been issued
      int sel_i;
      bool finite;
      warp_topk_select<8>(a.logits + static_cast<size_t>(warp) * a.E, a.E, a.k, lane, sel_i, sel_v, finite);
      if (bookkeeper && !finite && lane == 0) record_status(a.status, MOE_ERR_NONFINITE);
      if (lane < a.k) s_ids[warp * a.k + lane] = sel_i;
    } else {
      for (int i = lane; i < a.k; i += 32) {
        s_ids[warp * a.k + i] = __ldg(a.ids + warp * a.k + i);
        s_w[warp * a.k + i] = __ldg(a.w + warp * a.k + i);
      }
    }
  } else {
    // the other warps stage x (bf16 -> fp32) and its per-group sums
    constexpr int kStagers = kThreads - 32 * kGemvMaxT;
    const int n8 = kT * d / 8;
    for (int f = threadIdx.x - 32 * kGemvMaxT; f >= 0 && f < n8; f += kStagers) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.X) + f);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float4* d4 = reinterpret_cast<float4*>(xs + f * 8);
      d4[0] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                          __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
      d4[1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                          __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
    }
    if (warp >= kGemvMaxT) {
      asm volatile("bar.sync 1, %0;" ::"r"(kStagers) : "memory");  // the staging warps only
      for (int idx = warp - kGemvMaxT; idx < kT * 2 * L.KB1; idx += kWarps - kGemvMaxT) {
        float v = xs[(idx / (2 * L.KB1)) * d + (idx % (2 * L.KB1)) * 32 + lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) sx[idx] = v;
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // Distinct experts of the call in order of first appearance, and the
    // routing weight of each for each token.
    int nsl = rs0;
    if (kT == 1 && fused) {
      // one token: its k experts are distinct, slot j holds selection j
      if (lane < na) {
        slot_e[rs0 + lane] = s_ids[lane];
        s_slot[lane] = rs0 + lane;
      }
      nsl = rs0 + na;
    } else if (na <= 32) {
      // one assignment per lane: a lane whose expert no lower lane holds opens a slot
      const bool valid = lane < na;
      int e = valid ? s_ids[lane] : -1 - lane;
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
        s_slot[lane] = slot;
      }
      nsl = rs0 + __popc(opens);
    } else {
      // more assignments than lanes: walk them in order
      for (int i = 0; i < na; ++i) {
        int e = s_ids[i];
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
          s_slot[i] = slot;
        }
        __syncwarp();
      }
    }
    __syncwarp();
    if (lane == 0) {
      misc[0] = nsl - rs0;
      if (has_shared) slot_e[0] = 0;
    }
    __syncwarp();
    // the routed unit's loads start as soon as its expert is known
    const int U = Gs + (nsl - rs0) * G;
    if (u0 >= Gs && u0 < U) {
      const Unit m = unit_of(u0, Gs, G, has_shared);
      issue(m, slot_e[m.slot]);
    }
  }
  __syncthreads();
  const int U = Gs + misc[0] * G;
  pdl_launch_dependents();

  // The routing weights (fp64, slow on this GPU) are needed only from the down
  // projection on: warps < T compute them (and the weight of every slot)
  // while the other warps start on the gate/up products; warps < T take no
  // gate/up work.
  if (warp < kT) {
    if (fused) {
      const float w = warp_topk_weights(sel_v, a.k, lane);
      if (lane < a.k) s_w[warp * a.k + lane] = w;
    }
    asm volatile("bar.sync 3, %0;" ::"r"(32 * kT) : "memory");
    if (warp == 0) {
      for (int i = lane; i < na; i += 32) wt[s_slot[i] * kT + i / a.k] = s_w[i];
      if (has_shared && lane < kT) wt[lane] = 1.0f;
    }
  }
  if (bookkeeper) {
    asm volatile("bar.sync 2, %0;" ::"r"(kThreads) : "memory");  // the weights are in s_w
    // every routing output, as the routing kernel writes it for one chunk:
    // ids and weights, counts, exclusive offsets, the stable permutation and
    // the tile block map (experts ascending)
    int* cnt = reinterpret_cast<int*>(smem + L.qgu);  // [E]
    int* off = cnt + a.E;                              // [E + 1]
    int* boff = off + a.E + 1;                         // [E + 1]
    for (int i = threadIdx.x; i < na; i += kThreads) {
      a.out.ids[i] = s_ids[i];
      a.out.w[i] = s_w[i];
    }
    for (int e = threadIdx.x; e < a.E; e += kThreads) cnt[e] = 0;
    __syncwarp();
    asm volatile("bar.sync 2, %0;" ::"r"(kThreads) : "memory");
    for (int i = threadIdx.x; i < na; i += kThreads) atomicAdd(&cnt[s_ids[i]], 1);
    asm volatile("bar.sync 2, %0;" ::"r"(kThreads) : "memory");
    if (warp == 0) {
      int run = 0, brun = 0;
      for (int e0 = 0; e0 < a.E; e0 += 32) {
        const int e = e0 + lane;
        const int c = e < a.E ? cnt[e] : 0;
        const int b = (c + a.block_rows - 1) / a.block_rows;
        int ic = c, ib = b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int c2 = __shfl_up_sync(0xffffffffu, ic, o);
          const int b2 = __shfl_up_sync(0xffffffffu, ib, o);
          if (lane >= o) {
            ic += c2;
            ib += b2;
          }
        }
        if (e < a.E) {
          off[e] = run + ic - c;
          boff[e] = brun + ib - b;
        }
        run += __shfl_sync(0xffffffffu, ic, 31);
        brun += __shfl_sync(0xffffffffu, ib, 31);
      }
      if (lane == 0) {
        off[a.E] = run;
        boff[a.E] = brun;
        *a.out.num_blocks = brun;
      }
    }
    asm volatile("bar.sync 2, %0;" ::"r"(kThreads) : "memory");
    for (int e = threadIdx.x; e < a.E; e += kThreads) a.out.counts[e] = cnt[e];
    for (int e = threadIdx.x; e <= a.E; e += kThreads) a.out.offsets[e] = off[e];
    for (int i = threadIdx.x; i < na; i += kThreads) {
      const int e = s_ids[i];
      int r = 0;
      for (int j = 0; j < i; ++j) r += s_ids[j] == e;
      const int pos = off[e] + r;
      a.out.perm[pos] = i;
      a.out.inv_perm[i] = pos;
    }
    for (int e = threadIdx.x; e < a.E; e += kThreads) {
      const int c = cnt[e];
      int b = boff[e];
      for (int r = 0; r < c; r += a.block_rows, ++b) {
        a.out.block_map[3 * b + 0] = e;
        a.out.block_map[3 * b + 1] = off[e] + r;
        a.out.block_map[3 * b + 2] = min(a.block_rows, c - r);
      }
    }
  }

  const int p = threadIdx.x >> 1;  // down rows p, p + 256, ... of this CTA's half
  const int hf = threadIdx.x & 1;  // which 32 of the group's 64 columns
  uint32_t par = 0;
  int buf = 0;
  bool waited = false;
  bool ok = true;
  for (int u = u0; u < U; u += ncl) {
    const Unit m = unit_of(u, Gs, G, has_shared);
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar_h[buf], static_cast<uint32_t>(kT * (kRows + 1) * 4));
    // ---------------------------------------------------- gate/up: lane = row, warp = K slice
    float ag[kT], au[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) ag[t] = au[t] = 0.0f;
    // work item i = (group i/2, half i%2); warp w >= T takes items w-T,
    // w-T + (16-T), ...: the warps work on each chunk of codes as it lands
    ok &= mbar_wait_poll(bar_sb, par);
    for (int i = warp - kT; warp >= kT && i < 2 * L.KB1; i += kWarps - kT) {
      const int kb = i >> 1, hh = i & 1;
      ok &= mbar_wait_poll(&bar_gu[kb / kChunkGroups], par);
      half_group_dot2<kT>(qg, qu, lane, kb, hh, xs, d, sx, 2 * L.KB1, sbg[kb * kRows + lane], sbu[kb * kRows + lane],
                          ag, au);
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
      // token t = warp: h of this CTA's 32 features, into both CTAs; the copy
      // to the other CTA completes its exchange barrier
      const int t = warp;
      float g = 0.0f, uu = 0.0f;
#pragma unroll
      for (int s = 0; s < kWarps; ++s) {
        g += red[(s * kRows + lane) * kT + t];
        uu += red[((kWarps + s) * kRows + lane) * kT + t];
      }
      const float h = g / (1.0f + expf(-g)) * uu;
      const uint32_t peer = rank ^ 1u;
      const uint32_t peer_bar = mapa_shared(smem_u32(&bar_h[buf]), peer);
      float* dst = hbb + t * 64 + static_cast<int>(rank) * kRows + lane;
      *dst = h;
      st_async_f32(mapa_shared(smem_u32(dst), peer), h, peer_bar);
      // and the sum of these 32 values (the group sum of h needs both halves)
      float hsum_part = h;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) hsum_part += __shfl_xor_sync(0xffffffffu, hsum_part, off);
      if (lane == 0) {
        float* sdst = hsb + (buf * kT + t) * 2 + static_cast<int>(rank);
        *sdst = hsum_part;
        st_async_f32(mapa_shared(smem_u32(sdst), peer), hsum_part, peer_bar);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_h[buf]);  // this CTA's own half is written
    }
    ok &= mbar_wait_poll(&bar_h[buf], (static_cast<uint32_t>(u - u0) / static_cast<uint32_t>(ncl) >> 1) & 1u);
    // ---------------------------------------------------- down: thread pair = row, 32 columns each
    float wts[kT], hs[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      wts[t] = wt[m.slot * kT + t];
      hs[t] = hsb[(buf * kT + t) * 2] + hsb[(buf * kT + t) * 2 + 1];  // same order in both CTAs
    }
    for (int b = 0; b < L.nboxd; ++b) ok &= mbar_wait_poll(&bar_d[b], par);
    const float* hp = hbb + hf * 32;
    // two rows at a time: independent dependency chains
    for (int row0 = p; row0 < L.half; row0 += 2 * kPairs) {
      const int row1 = row0 + kPairs;
      const bool has1 = row1 < L.half;
      float2 pp0[kT], pp1[kT];
#pragma unroll
      for (int t = 0; t < kT; ++t) pp0[t] = pp1[t] = make_float2(0.0f, 0.0f);
      const uint4 w0 = *reinterpret_cast<const uint4*>(qd + row0 * 32 + hf * 16);
      const uint4 w1 = has1 ? *reinterpret_cast<const uint4*>(qd + row1 * 32 + hf * 16) : make_uint4(0, 0, 0, 0);
      word_dot<kT>(w0.x, hp + 0, 64, pp0);
      word_dot<kT>(w1.x, hp + 0, 64, pp1);
      word_dot<kT>(w0.y, hp + 8, 64, pp0);
      word_dot<kT>(w1.y, hp + 8, 64, pp1);
      word_dot<kT>(w0.z, hp + 16, 64, pp0);
      word_dot<kT>(w1.z, hp + 16, 64, pp1);
      word_dot<kT>(w0.w, hp + 24, 64, pp0);
      word_dot<kT>(w1.w, hp + 24, 64, pp1);
      const uint32_t sb0 = sbd[row0];
      const uint32_t sb1 = has1 ? sbd[row1] : 0u;
      const float s0 = __uint_as_float(sb0 << 16), s1 = __uint_as_float(sb1 << 16);
      const float c0 = __uint_as_float(sb0 & 0xFFFF0000u) - 128.0f * s0;
      const float c1 = __uint_as_float(sb1 & 0xFFFF0000u) - 128.0f * s1;
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        float pv0 = pp0[t].x + pp0[t].y;
        float pv1 = pp1[t].x + pp1[t].y;
        pv0 += __shfl_xor_sync(0xffffffffu, pv0, 1);
        pv1 += __shfl_xor_sync(0xffffffffu, pv1, 1);
        if (hf == 0 && wts[t] != 0.0f) {
          accd[row0 * kT + t] = fmaf(wts[t], fmaf(s0, pv0, c0 * hs[t]), accd[row0 * kT + t]);
          if (has1) accd[row1 * kT + t] = fmaf(wts[t], fmaf(s1, pv1, c1 * hs[t]), accd[row1 * kT + t]);
        }
      }
    }
    __syncthreads();  // every box of this unit has been read
    if (u + ncl < U && warp == 0) {
      const Unit nx = unit_of(u + ncl, Gs, G, has_shared);
      issue(nx, nx.shared ? 0 : slot_e[nx.slot]);
    }
    par ^= 1;
    buf ^= 1;
  }
  if (!waited) cluster_wait();
  if (!ok) record_status(a.status, MOE_ERR_TIMEOUT);

  // ---------------------------------------------------- Y: partial rows, one grid barrier, every CTA sums a few rows
  // This cluster's share of the output (rows of this CTA's half; zeros for a
  // CTA with no unit) goes to global memory.  After a barrier over the grid
  // (bounded spin on an arrival counter; every CTA of the launch is resident,
  // one per SM), CTA b sums the partials of rows [b*per, (b+1)*per) over the
  // clusters in a fixed order, so the result does not depend on timing.
  {
    float* part = a.part + static_cast<size_t>(cl) * kT * d + static_cast<int>(rank) * L.half;
    for (int i = threadIdx.x; i < L.half * kT; i += kThreads) {
      const int t = i / L.half, row = i % L.half;
      part[static_cast<size_t>(t) * d + row] = accd[row * kT + t];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    atom_add_acq_rel_gpu(&hdr->dec_arrive, 1u);
    const long long t0 = clock64();
    while (ld_acquire_gpu(&hdr->dec_arrive) < gridDim.x) {
      if (clock64() - t0 > kWaitLimitCycles) {
        record_status(a.status, MOE_ERR_TIMEOUT);
        break;
      }
      __nanosleep(20);
    }
  }
  __syncthreads();
  {
    const int nclu = static_cast<int>(gridDim.x >> 1);
    const int per = (d + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int r0 = static_cast<int>(blockIdx.x) * per;
    const int r1 = min(d, r0 + per);
    const int items = max(0, r1 - r0) * kT;
    // S threads per output value, S a power of two <= 32 (lanes of one warp)
    int S = 1;
    while (S < 32 && items * S * 2 <= kThreads) S *= 2;
    const int j = threadIdx.x % S;
    for (int it = threadIdx.x / S; it < (items + (kThreads / S) - 1) / (kThreads / S) * (kThreads / S); it += kThreads / S) {
      float v = 0.0f;
      int t = 0, row = 0;
      if (it < items) {
        t = it / (r1 - r0);
        row = r0 + it % (r1 - r0);
        // four loads in flight per round, added in cluster order
        for (int c0 = j; c0 < nclu; c0 += 4 * S) {
          float pv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = c0 + q * S;
            pv[q] = c < nclu ? __ldcg(a.part + (static_cast<size_t>(c) * kT + t) * d + row) : 0.0f;
          }
          v += pv[0];
          v += pv[1];
          v += pv[2];
          v += pv[3];
        }
      }
      for (int off = 1; off < S; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (it < items && j == 0) a.Y[static_cast<size_t>(t) * d + row] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // the last CTA out resets the counters for the next call (all have passed the barrier)
    if (atom_add_acq_rel_gpu(&hdr->dec_done, 1u) == gridDim.x - 1) {
      hdr->dec_arrive = 0;
      hdr->dec_done = 0;
      __threadfence();
    }
  }
}

// Clusters of this kernel that can be resident at once on the current device
// (0 on error).  The kernel's grid barrier needs every CTA resident together.
template <int kT>
int max_clusters(size_t smem) {
  static int cached_dev = -1, cached = 0;
  static size_t cached_smem = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev == cached_dev && smem == cached_smem) return cached;
  if (cudaFuncSetAttribute(decode_kernel<kT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
      cudaSuccess)
    return 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<kT>, &cfg) != cudaSuccess) return 0;
  cached_dev = dev;
  cached_smem = smem;
  cached = n;
  return n;
}

template <int kT>
cudaError_t launch_t(const DecodeArgs& a, const DecodeMaps* routed, const DecodeMaps* sh, WsHeader* hdr, int ncl,
                     size_t smem, cudaStream_t stream, bool pdl) {
  const int resident = max_clusters<kT>(smem);
  if (resident < 1 + (a.logits ? 1 : 0)) return cudaErrorInvalidConfiguration;
  if (ncl > resident) ncl = resident;
  const int grid = 2 * ncl;
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
  // the routing outputs' scratch (counts and two scans over E <= 256) reuses the gate/up code buffer
  if (2ull * L.nchunk * kChunkGroups * kRows * 32 < 3ull * 257 * 4) return false;
  return L.total <= 227 * 1024 && L.nchunk + 1 + L.nboxd <= 32 && d % 64 == 0 && I % 64 == 0 &&
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
  const int extra = a.logits ? 1 : 0;  // the cluster that writes the routing outputs
  int ncl = a.num_sms / 2 - extra;
  if (ncl > units) ncl = units;
  if (ncl > kDecodeMaxClusters - extra) ncl = kDecodeMaxClusters - extra;
  if (ncl < 1) ncl = 1;
  ncl += extra;  // capped below by the clusters that fit on the device at once
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  timer_begin(kKDecode, stream);
  cudaError_t err;
  switch (a.T) {
    case 1: err = launch_t<1>(a, routed, sh, hdr, ncl, L.total, stream, pdl); break;
    case 2: err = launch_t<2>(a, routed, sh, hdr, ncl, L.total, stream, pdl); break;
    case 3: err = launch_t<3>(a, routed, sh, hdr, ncl, L.total, stream, pdl); break;
    default: err = launch_t<4>(a, routed, sh, hdr, ncl, L.total, stream, pdl); break;
  }
  timer_end(kKDecode, stream);
  return err;
}

}  // namespace bm
