// Decode path (small T): the expert projections as matrix-vector products on
// the CUDA cores.  "Perplexity's Lily Beats MLX-LM on MacBook M5", section
// "Prefill and decode are different problems": batch-1 decode is a GEMV bound
// by memory bandwidth that belongs on the vector ALUs; section "Decode:
// minimize bytes per token": the expert input projections are fused with the
// gate activation, and the output projection with the routing scores and the
// shared expert.
//
// Design (sm_103a): each CTA owns a tile of weight rows of one (token, expert)
// pair and issues, up front, TMA loads of every byte it needs -- codes and
// group parameters -- so each active expert's bytes cross HBM exactly once and
// a whole CTA's share is in flight at the same time.  A thread owns one row and
// a slice of K; the token vector is broadcast from shared memory.  The 4-bit
// codes become fp32 values 128+q with one byte permute each (exponent of 128,
// code in the low mantissa bits), are multiplied by x with packed fp32x2 FMAs,
// and the affine map is applied once per 64-column group:
//   sum_k (q_k s + b) x_k = s * sum_k (128+q_k) x_k + (b - 128 s) * sum_k x_k.
// Two kernels per layer: gate/up + SwiGLU -> h (fp32), then down + weighted
// combine + shared expert -> Y (bf16).  They chain with programmatic dependent
// launch: the down kernel's weight loads start while the gate/up kernel runs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bm {

namespace {

constexpr int kGUThreads = 512;  // lane = row (32 rows), warp = K slice (16 slices)
constexpr int kGUSlices = kGUThreads / 32;
constexpr int kDownThreads = 256;  // 16 rows x 16 work slices
constexpr int kDownSlices = kDownThreads / kGemvRowsDown;
constexpr uint32_t kMagic128 = 0x43000000u;  // fp32 128.0: a code in bits 16..19 reads as 128 + q
constexpr int kBoxWords = 32;                // 128-byte rows per TMA box
constexpr int kBoxKB = 4;                    // 64-column groups per box row

__host__ __device__ constexpr int div_up(int a, int b) { return (a + b - 1) / b; }

// sum over 8 codes of one word of (128 + q) * x, accumulated in a pair.
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
//   tile:  the TMA box holding the row (128-byte rows, 128-byte swizzle)
//   row:   row inside the box; kb: group index (selects the 32-byte chunk pair)
//   xg:    the 64 fp32 x values of this group (shared memory, broadcast)
__device__ __forceinline__ float group_dot(const uint8_t* tile, int row, int kb, const float* xg, float sx,
                                           uint32_t sbv) {
  const int c0 = ((kb & 3) * 2) ^ (row & 7);
  const int c1 = ((kb & 3) * 2 + 1) ^ (row & 7);
  const uint4 wa = *reinterpret_cast<const uint4*>(tile + row * 128 + c0 * 16);
  const uint4 wb = *reinterpret_cast<const uint4*>(tile + row * 128 + c1 * 16);
  const float4* x4 = reinterpret_cast<const float4*>(xg);
  float2 acc = make_float2(0.0f, 0.0f);
  acc = codes_dot8(wa.x, x4[0], x4[1], acc);
  acc = codes_dot8(wa.y, x4[2], x4[3], acc);
  acc = codes_dot8(wa.z, x4[4], x4[5], acc);
  acc = codes_dot8(wa.w, x4[6], x4[7], acc);
  acc = codes_dot8(wb.x, x4[8], x4[9], acc);
  acc = codes_dot8(wb.y, x4[10], x4[11], acc);
  acc = codes_dot8(wb.z, x4[12], x4[13], acc);
  acc = codes_dot8(wb.w, x4[14], x4[15], acc);
  const float s = __uint_as_float(sbv << 16);
  const float b = __uint_as_float(sbv & 0xFFFF0000u);
  return fmaf(s, acc.x + acc.y, (b - 128.0f * s) * sx);
}

// Loads x (bf16 [K]) into shared memory as fp32 and the per-group sums.
__device__ __forceinline__ void stage_vector_bf16(const uint16_t* __restrict__ src, int K, float* xs, float* sxs) {
  for (int c = threadIdx.x * 2; c < K; c += blockDim.x * 2) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(src + c);
    xs[c] = __uint_as_float(v << 16);
    xs[c + 1] = __uint_as_float(v & 0xFFFF0000u);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int kb = warp; kb < K / 64; kb += blockDim.x / 32) {
    float v = xs[kb * 64 + lane] + xs[kb * 64 + 32 + lane];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) sxs[kb] = v;
  }
}

struct GUSmem {
  int nbox, KB;
  size_t q_off, sb_off, x_off, sx_off, red_off, bar_off, total;
};

__host__ __device__ inline GUSmem gu_layout(int K) {
  GUSmem L;
  L.KB = K / 64;
  L.nbox = div_up(K / 8, kBoxWords);
  size_t o = 0;
  L.q_off = o;
  o += 2ull * L.nbox * kGemvRowsGU * 128;  // gate then up
  L.sb_off = o;  // 1024-aligned; the up matrix's block starts KB*128 bytes later (128-aligned)
  o += 2ull * L.KB * kGemvRowsGU * 4;
  L.x_off = o;
  o += static_cast<size_t>(K) * 4;
  L.sx_off = o;
  o += static_cast<size_t>(L.KB) * 4;
  o = (o + 15) & ~static_cast<size_t>(15);
  L.red_off = o;
  o += 2ull * kGUSlices * 32 * 4;
  L.bar_off = o;
  o += static_cast<size_t>(L.nbox + 1) * 8;
  L.total = o + 1024;  // alignment slack
  return L;
}

__global__ void __launch_bounds__(kGUThreads, 1)
    gemv_gateup_kernel(const __grid_constant__ CUtensorMap qg_r, const __grid_constant__ CUtensorMap qu_r,
                       const __grid_constant__ CUtensorMap sbg_r, const __grid_constant__ CUtensorMap sbu_r,
                       const __grid_constant__ CUtensorMap qg_s, const __grid_constant__ CUtensorMap qu_s,
                       const __grid_constant__ CUtensorMap sbg_s, const __grid_constant__ CUtensorMap sbu_s,
                       GemvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int pair = blockIdx.y;
  const int routed_pairs = a.T * a.k;
  const bool is_shared = pair >= routed_pairs;
  const int Icur = is_shared ? a.I_shared : a.I;
  const int n0 = blockIdx.x * kGemvRowsGU;
  if (n0 >= Icur) return;
  const int K = a.d;
  const GUSmem L = gu_layout(K);
  const int t = is_shared ? pair - routed_pairs : pair / a.k;

  uint8_t* qg = smem + L.q_off;
  uint8_t* qu = qg + static_cast<size_t>(L.nbox) * kGemvRowsGU * 128;
  uint32_t* sbg = reinterpret_cast<uint32_t*>(smem + L.sb_off);
  uint32_t* sbu = sbg + L.KB * kGemvRowsGU;
  float* xs = reinterpret_cast<float*>(smem + L.x_off);
  float* sxs = reinterpret_cast<float*>(smem + L.sx_off);
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);

  const CUtensorMap* mqg = is_shared ? &qg_s : &qg_r;
  const CUtensorMap* mqu = is_shared ? &qu_s : &qu_r;
  const CUtensorMap* msbg = is_shared ? &sbg_s : &sbg_r;
  const CUtensorMap* msbu = is_shared ? &sbu_s : &sbu_r;

  if (threadIdx.x == 0) {
    for (int b = 0; b <= L.nbox; ++b) mbar_init(&bars[b], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Lane b < nbox of warp 0 loads code box b of both matrices; lane nbox the
  // group parameters.
  auto issue_loads = [&](int e) {
    const uint32_t box_bytes = kGemvRowsGU * 128;
    const int b = threadIdx.x;
    if (b < L.nbox) {
      mbar_arrive_expect_tx(&bars[b], 2 * box_bytes);
      tma_load_3d(qg + static_cast<size_t>(b) * box_bytes, mqg, &bars[b], b * kBoxWords, n0, e);
      tma_load_3d(qu + static_cast<size_t>(b) * box_bytes, mqu, &bars[b], b * kBoxWords, n0, e);
    } else if (b == L.nbox) {
      mbar_arrive_expect_tx(&bars[L.nbox], 2u * L.KB * kGemvRowsGU * 4);
      tma_load_3d(sbg, msbg, &bars[L.nbox], n0, 0, e);
      tma_load_3d(sbu, msbu, &bars[L.nbox], n0, 0, e);
    }
  };

  // The shared expert's weights do not depend on the previous kernel.
  if (threadIdx.x <= L.nbox && is_shared) issue_loads(0);
  pdl_wait();
  if (threadIdx.x <= L.nbox && !is_shared) {
    int e = a.ids[pair];
    if (e < 0 || e >= a.E) {
      record_status(a.status, MOE_ERR_INVALID_ARG);
      e = 0;
    }
    issue_loads(e);
  }
  pdl_launch_dependents();

  stage_vector_bf16(a.X + static_cast<size_t>(t) * K, K, xs, sxs);
  __syncthreads();

  const int r = threadIdx.x & 31;
  const int ks = threadIdx.x >> 5;
  float acc_g = 0.0f, acc_u = 0.0f;
  bool ok = mbar_wait(&bars[L.nbox], 0, nullptr);
  for (int kb = ks; kb < L.KB; kb += kGUSlices) {
    const int b = kb / kBoxKB;
    ok &= mbar_wait(&bars[b], 0, nullptr);
    const size_t boff = static_cast<size_t>(b) * kGemvRowsGU * 128;
    const float* xg = xs + kb * 64;
    acc_g += group_dot(qg + boff, r, kb, xg, sxs[kb], sbg[kb * kGemvRowsGU + r]);
    acc_u += group_dot(qu + boff, r, kb, xg, sxs[kb], sbu[kb * kGemvRowsGU + r]);
  }
  if (!ok) record_status(a.status, MOE_ERR_TIMEOUT);
  red[ks * 32 + r] = acc_g;
  red[kGUSlices * 32 + ks * 32 + r] = acc_u;
  __syncthreads();
  if (ks == 0) {
    float g = 0.0f, u = 0.0f;
#pragma unroll
    for (int s = 0; s < kGUSlices; ++s) {
      g += red[s * 32 + r];
      u += red[kGUSlices * 32 + s * 32 + r];
    }
    const float h = g / (1.0f + expf(-g)) * u;
    float* dst = is_shared ? a.h_shared + static_cast<size_t>(t) * a.I_shared
                           : a.h_routed + static_cast<size_t>(pair) * a.I;
    dst[n0 + r] = h;
  }
}

struct DownSmem {
  int nbox_r, nbox_s, KB_r, KB_s, nexp, Imax;
  size_t sb_slot_r;  // bytes per routed expert's group parameters, rounded to 128 (TMA destination)
  size_t q_off, q_s_off, sb_off, sb_s_off, h_off, sx_off, w_off, red_off, bar_off, total;
};

__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Every TMA destination starts on a 1024-byte boundary (128-byte swizzled code
// boxes) or a 128-byte boundary (group parameters).
__host__ __device__ inline DownSmem down_layout(int I, int I_shared, int k) {
  DownSmem L;
  L.KB_r = I / 64;
  L.KB_s = I_shared / 64;
  L.nbox_r = div_up(I / 8, kBoxWords);
  L.nbox_s = I_shared > 0 ? div_up(I_shared / 8, kBoxWords) : 0;
  L.nexp = k + (I_shared > 0 ? 1 : 0);
  L.Imax = I > I_shared ? I : I_shared;
  L.sb_slot_r = round_up(static_cast<size_t>(L.KB_r) * kGemvRowsDown * 4, 128);
  const size_t box = kGemvRowsDown * 128;
  size_t o = 0;
  L.q_off = o;
  o += static_cast<size_t>(k) * L.nbox_r * box;
  L.q_s_off = o;
  o += static_cast<size_t>(L.nbox_s) * box;
  L.sb_off = o;
  o += static_cast<size_t>(k) * L.sb_slot_r;
  L.sb_s_off = o;
  o += round_up(static_cast<size_t>(L.KB_s) * kGemvRowsDown * 4, 128);
  L.h_off = o;
  o += static_cast<size_t>(L.nexp) * L.Imax * 4;
  L.sx_off = o;
  o += static_cast<size_t>(L.nexp) * (L.Imax / 64) * 4;
  L.w_off = o;
  o += static_cast<size_t>(L.nexp) * 4;
  o = round_up(o, 16);
  L.red_off = o;
  o += static_cast<size_t>(kDownSlices) * kGemvRowsDown * 4;
  L.bar_off = o;
  o += static_cast<size_t>(L.nexp) * 8;
  L.total = o + 1024;
  return L;
}

__global__ void __launch_bounds__(kDownThreads, 1)
    gemv_down_kernel(const __grid_constant__ CUtensorMap qd_r, const __grid_constant__ CUtensorMap sbd_r,
                     const __grid_constant__ CUtensorMap qd_s, const __grid_constant__ CUtensorMap sbd_s,
                     GemvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int t = blockIdx.y;
  const int n0 = blockIdx.x * kGemvRowsDown;
  const int k = a.k;
  const DownSmem L = down_layout(a.I, a.I_shared, k);
  const size_t box = kGemvRowsDown * 128;
  const bool has_shared = a.I_shared > 0;

  uint8_t* q_r = smem + L.q_off;
  uint8_t* q_s = smem + L.q_s_off;
  uint32_t* sb_s = reinterpret_cast<uint32_t*>(smem + L.sb_s_off);
  float* hs = reinterpret_cast<float*>(smem + L.h_off);
  float* sxs = reinterpret_cast<float*>(smem + L.sx_off);
  float* ws = reinterpret_cast<float*>(smem + L.w_off);
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);

  if (threadIdx.x == 0) {
    for (int j = 0; j < L.nexp; ++j) mbar_init(&bars[j], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Lane j of warp 0 loads expert j's codes and group parameters (lane k: the
  // shared expert).  The routing was complete before the gate/up kernel
  // released this grid, so the expert ids can be read before waiting on that
  // kernel; only h needs the wait.
  if (threadIdx.x < L.nexp) {
    const int j = threadIdx.x;
    if (j == k) {
      mbar_arrive_expect_tx(&bars[k], static_cast<uint32_t>(L.nbox_s * box + L.KB_s * kGemvRowsDown * 4));
      tma_load_3d(sb_s, &sbd_s, &bars[k], n0, 0, 0);
      for (int b = 0; b < L.nbox_s; ++b) tma_load_3d(q_s + b * box, &qd_s, &bars[k], b * kBoxWords, n0, 0);
    } else {
      int e = a.ids[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= a.E) {
        record_status(a.status, MOE_ERR_INVALID_ARG);
        e = 0;
      }
      uint8_t* qj = q_r + static_cast<size_t>(j) * L.nbox_r * box;
      uint32_t* sbj = reinterpret_cast<uint32_t*>(smem + L.sb_off + static_cast<size_t>(j) * L.sb_slot_r);
      mbar_arrive_expect_tx(&bars[j], static_cast<uint32_t>(L.nbox_r * box + L.KB_r * kGemvRowsDown * 4));
      tma_load_3d(sbj, &sbd_r, &bars[j], n0, 0, e);
      for (int b = 0; b < L.nbox_r; ++b) tma_load_3d(qj + b * box, &qd_r, &bars[j], b * kBoxWords, n0, e);
    }
  }
  pdl_wait();  // h from the gate/up kernel
  pdl_launch_dependents();

  // stage h (fp32) of every expert of this token, its group sums, and weights
  for (int j = 0; j < L.nexp; ++j) {
    const bool sh = j == k;
    const int Ij = sh ? a.I_shared : a.I;
    const float* src = sh ? a.h_shared + static_cast<size_t>(t) * a.I_shared
                          : a.h_routed + (static_cast<size_t>(t) * k + j) * a.I;
    float* dst = hs + static_cast<size_t>(j) * L.Imax;
    for (int c = threadIdx.x * 4; c < Ij; c += kDownThreads * 4)
      *reinterpret_cast<float4*>(dst + c) = *reinterpret_cast<const float4*>(src + c);
  }
  if (threadIdx.x < k) ws[threadIdx.x] = a.w[static_cast<size_t>(t) * k + threadIdx.x];
  if (threadIdx.x == 0 && has_shared) ws[k] = 1.0f;
  __syncthreads();
  {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gpe = L.Imax / 64;
    for (int id = warp; id < L.nexp * gpe; id += kDownThreads / 32) {
      const int j = id / gpe, kb = id % gpe;
      const int Ij = (j == k) ? a.I_shared : a.I;
      if (kb * 64 >= Ij) continue;
      const float* x = hs + static_cast<size_t>(j) * L.Imax + kb * 64;
      float v = x[lane] + x[32 + lane];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) sxs[j * gpe + kb] = v;
    }
  }
  __syncthreads();

  const int r = threadIdx.x % kGemvRowsDown;
  const int slice = threadIdx.x / kGemvRowsDown;
  const int gpe = L.Imax / 64;
  const int P = k * L.KB_r + (has_shared ? L.KB_s : 0);
  float acc = 0.0f;
  bool ok = true;
  for (int p = slice; p < P; p += kDownSlices) {
    int j, kb;
    if (p < k * L.KB_r) {
      j = p / L.KB_r;
      kb = p % L.KB_r;
    } else {
      j = k;
      kb = p - k * L.KB_r;
    }
    ok &= mbar_wait(&bars[j], 0, nullptr);
    const uint8_t* tile;
    uint32_t sbv;
    if (j < k) {
      tile = q_r + (static_cast<size_t>(j) * L.nbox_r + kb / kBoxKB) * box;
      sbv = reinterpret_cast<const uint32_t*>(smem + L.sb_off + static_cast<size_t>(j) * L.sb_slot_r)
          [kb * kGemvRowsDown + r];
    } else {
      tile = q_s + static_cast<size_t>(kb / kBoxKB) * box;
      sbv = sb_s[kb * kGemvRowsDown + r];
    }
    const float d = group_dot(tile, r, kb, hs + static_cast<size_t>(j) * L.Imax + kb * 64, sxs[j * gpe + kb], sbv);
    acc = fmaf(ws[j], d, acc);
  }
  // every expert's barrier must have completed before the CTA may exit
  for (int j = threadIdx.x; j < L.nexp; j += kDownThreads) ok &= mbar_wait(&bars[j], 0, nullptr);
  if (!ok) record_status(a.status, MOE_ERR_TIMEOUT);
  red[slice * kGemvRowsDown + r] = acc;
  __syncthreads();
  if (slice == 0) {
    float y = 0.0f;
#pragma unroll
    for (int s = 0; s < kDownSlices; ++s) y += red[s * kGemvRowsDown + r];
    a.Y[static_cast<size_t>(t) * a.d + n0 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  }
}

bool g_attr_set = false;

}  // namespace

size_t gemv_smem_gateup(int d) { return gu_layout(d).total; }
size_t gemv_smem_down(int I, int I_shared, int k) { return down_layout(I, I_shared, k).total; }

cudaError_t launch_gemv(const GemvArgs& a, const GemvMaps* routed, const GemvMaps* shared, cudaStream_t stream,
                        bool pdl) {
  const GUSmem Lg = gu_layout(a.d);
  const DownSmem Ld = down_layout(a.I, a.I_shared, a.k);
  // TMA destinations: swizzled code boxes on 1024 bytes, group parameters on 128
  const bool aligned = Lg.q_off % 1024 == 0 && (static_cast<size_t>(Lg.nbox) * kGemvRowsGU * 128) % 1024 == 0 &&
                       Lg.sb_off % 128 == 0 && (static_cast<size_t>(Lg.KB) * kGemvRowsGU * 4) % 128 == 0 &&
                       Ld.q_off % 1024 == 0 && Ld.q_s_off % 1024 == 0 && Ld.sb_off % 128 == 0 &&
                       Ld.sb_slot_r % 128 == 0 && Ld.sb_s_off % 128 == 0 && Lg.bar_off % 8 == 0 &&
                       Ld.bar_off % 8 == 0;
  if (!aligned) return cudaErrorInvalidValue;
  if (!g_attr_set) {
    cudaError_t e1 = cudaFuncSetAttribute(gemv_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaError_t e2 = cudaFuncSetAttribute(gemv_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e1 != cudaSuccess) return e1;
    if (e2 != cudaSuccess) return e2;
    g_attr_set = true;
  }
  const GemvMaps* sh = shared ? shared : routed;  // unused when there is no shared expert
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int Imax = a.I > a.I_shared ? a.I : a.I_shared;
  cfg.gridDim = dim3(div_up(Imax, kGemvRowsGU), a.T * a.k + (a.I_shared > 0 ? a.T : 0));
  cfg.blockDim = dim3(kGUThreads);
  cfg.dynamicSmemBytes = Lg.total;
  timer_begin(kKGemvGateUp, stream);
  cudaError_t err = cudaLaunchKernelEx(&cfg, gemv_gateup_kernel, routed->q_gate, routed->q_up, routed->sb_gate,
                                       routed->sb_up, sh->q_gate, sh->q_up, sh->sb_gate, sh->sb_up, a);
  timer_end(kKGemvGateUp, stream);
  if (err != cudaSuccess) return err;

  cfg.gridDim = dim3(a.d / kGemvRowsDown, a.T);
  cfg.blockDim = dim3(kDownThreads);
  cfg.dynamicSmemBytes = Ld.total;
  attr[0].val.programmaticStreamSerializationAllowed = 1;  // always chained to the gate/up kernel
  timer_begin(kKGemvDown, stream);
  err = cudaLaunchKernelEx(&cfg, gemv_down_kernel, routed->q_down, routed->sb_down, sh->q_down, sh->sb_down, a);
  timer_end(kKGemvDown, stream);
  return err;
}

}  // namespace bm
