// Router projection: logits[t][e] = sum_i X[t][i] * Wr[e][i], bf16 operands,
// fp32 accumulation ("Perplexity's Lily Beats MLX-LM on MacBook M5", section
// "Why Qwen3.6-35B-A3B is a weird workload": the router scores each of the 256
// experts for every token and picks 8; the score is read as a linear map of the
// token's hidden state, accumulated in fp32 like the pages' other products).
//
// Warp-level tensor-core MMAs (mma.sync m16n8k16, bf16 in, fp32 out) with the
// router rows as the M operand and the tokens as N, so one token (decode) still
// fills the rows of every MMA.  The operands are read straight from global
// memory, 16 bytes per lane, in a permuted K order that both operands share:
// lane (g, q) loads columns 8q .. 8q+7 of a 32-column chunk of its rows g and
// g+8 (router) and of its token g; the first MMA takes their pairs 0 and 1 as
// the fragment's columns (2q, 2q+1) and (2q+8, 2q+9), the second MMA pairs 2
// and 3.  Both operands use the same map from fragment column to K, so every
// product X[t][i] * Wr[e][i] is formed exactly once; the permutation changes
// only the order of the fp32 additions.
//
// Two shapes.  Up to 32 tokens: a warp per router row on the CUDA cores, each
// lane with its whole share of the row in flight at once (the rows stream
// from HBM once; the products of bf16 values are exact in fp32, each sum is
// rounded once per step); a lane's partial sums are combined across the warp
// in a fixed tree.  More tokens: the tensor-core MMAs below on a CTA tile of 32
// experts x 64 tokens; the tiles of each 128-wide K chunk are staged in shared
// memory with cp.async, four chunks in flight, so every byte is read from L2
// once per CTA, and each warp multiplies 16 experts x 16 tokens from there.
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bm {

namespace {

constexpr int kRouterThreads = 256;

// Up to kRowsMaxT tokens: warp w of CTA b computes router row 4b + w for
// every token.
constexpr int kRowsThreads = 128;
constexpr int kRowsMaxT = 32;
constexpr int kRowsU = 8;  // 16-byte pieces of the row per lane in flight (a 2048-wide row in one round)
constexpr int kRowsG = 4;  // tokens whose loads are in flight together

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b, float acc) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc = fmaf(__uint_as_float(av[j] << 16), __uint_as_float(bv[j] << 16), acc);
    acc = fmaf(__uint_as_float(av[j] & 0xFFFF0000u), __uint_as_float(bv[j] & 0xFFFF0000u), acc);
  }
  return acc;
}

__global__ void __launch_bounds__(kRowsThreads)
    router_rows_kernel(const uint16_t* __restrict__ X, int T, int d, const uint16_t* __restrict__ Wr, int E,
                       float* __restrict__ logits) {
  pdl_wait();  // X may come from the previous kernel on the stream
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * (kRowsThreads / 32) + (threadIdx.x >> 5);
  if (e >= E) return;
  const int n16 = d / 8;  // 16-byte pieces per row
  const uint4* w = reinterpret_cast<const uint4*>(Wr + static_cast<size_t>(e) * d);
  const uint4* xr = reinterpret_cast<const uint4*>(X);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  // tokens in groups of kRowsG, every load of a group in flight together (the
  // router row comes from HBM for the first group and from L1 after it)
  for (int t0 = 0; t0 < T; t0 += kRowsG) {
    float acc[kRowsG];
#pragma unroll
    for (int j = 0; j < kRowsG; ++j) acc[j] = 0.0f;
    for (int i0 = lane; i0 < n16; i0 += 32 * kRowsU) {
      uint4 wv[kRowsU], xv[kRowsG][kRowsU];
#pragma unroll
      for (int u = 0; u < kRowsU; ++u) {
        const bool in = i0 + 32 * u < n16;
        wv[u] = in ? __ldg(w + i0 + 32 * u) : zero;
#pragma unroll
        for (int j = 0; j < kRowsG; ++j)
          xv[j][u] = (in && t0 + j < T) ? __ldg(xr + static_cast<size_t>(t0 + j) * n16 + i0 + 32 * u) : zero;
      }
#pragma unroll
      for (int j = 0; j < kRowsG; ++j)
#pragma unroll
        for (int u = 0; u < kRowsU; ++u) acc[j] = dot8_bf16(wv[u], xv[j][u], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < kRowsG; ++j) {
      float v = acc[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t0 + j < T) logits[static_cast<size_t>(t0 + j) * E + e] = v;
    }
  }
}

// Shared-memory-staged shape: CTA tile kSE experts x kST tokens, K chunks of
// kSK.  A staged row is kSPitch bf16 (kSK used): 320 bytes, so the two rows a
// quarter-warp reads with 16-byte loads fall in opposite halves of the banks.
constexpr int kSE = 32, kST = 64, kSK = 128, kSPitch = 160;
constexpr int kSStages = 4;  // K chunks in flight
constexpr int kSStageElems = (kSE + kST) * kSPitch;
constexpr int kSSmemBytes = kSStages * kSStageElems * 2;

__global__ void __launch_bounds__(kRouterThreads)
    router_smem_kernel(const uint16_t* __restrict__ X, int T, int d, const uint16_t* __restrict__ Wr, int E,
                       float* __restrict__ logits) {
  extern __shared__ __align__(16) uint16_t s_stage[];  // [kSStages][router rows | token rows][kSPitch]

  pdl_wait();  // X may come from the previous kernel on the stream
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int wm = warp & 1, wn = warp >> 1;  // 16 experts x 16 tokens each
  const int e_base = blockIdx.x * kSE, t_base = blockIdx.y * kST;
  constexpr int kPieces = kSK / 8;                       // 16-byte pieces per staged row
  constexpr int kCopies = (kSE + kST) * kPieces;         // per stage
  static_assert(kCopies % kRouterThreads == 0, "whole copies per thread");

  auto stage = [&](int buf, int c) {  // every thread commits one group per call
#pragma unroll
    for (int i = 0; i < kCopies / kRouterThreads; ++i) {
      const int p = threadIdx.x + i * kRouterThreads;
      const int row = p / kPieces, piece = p % kPieces;
      uint16_t* dst = s_stage + buf * kSStageElems + row * kSPitch + 8 * piece;
      const int col = c * kSK + 8 * piece;  // past d (a chunk's second half when d % kSK = 64): zeros
      const bool kin = col < d;
      if (row < kSE) {
        const int e = e_base + row;
        cp_async16(dst, Wr + static_cast<size_t>(e < E ? e : 0) * d + (kin ? col : 0), e < E && kin);
      } else {
        const int t = t_base + row - kSE;
        cp_async16(dst, X + static_cast<size_t>(t < T ? t : 0) * d + (kin ? col : 0), t < T && kin);
      }
    }
    cp_async_commit();
  };

  float acc[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;

  // chunk c lives in stage c % kSStages; a commit group per chunk (empty past
  // the end), so waiting for all but the newest kSStages - 1 groups means
  // chunk c has landed
  const int nchunk = (d + kSK - 1) / kSK;
#pragma unroll
  for (int c = 0; c < kSStages - 1; ++c) {
    if (c < nchunk) stage(c, c);
    else cp_async_commit();
  }
  for (int c = 0; c < nchunk; ++c) {
    if (c + kSStages - 1 < nchunk) stage((c + kSStages - 1) % kSStages, c + kSStages - 1);
    else cp_async_commit();
    cp_async_wait<kSStages - 1>();
    __syncthreads();
    const uint16_t* w = s_stage + (c % kSStages) * kSStageElems;
    const uint16_t* x = w + kSE * kSPitch;
#pragma unroll
    for (int sub = 0; sub < kSK / 32; ++sub) {
      const int col = 32 * sub + 8 * q;
      const uint4 Ag = *reinterpret_cast<const uint4*>(w + (16 * wm + g) * kSPitch + col);
      const uint4 Ag8 = *reinterpret_cast<const uint4*>(w + (16 * wm + g + 8) * kSPitch + col);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint4 B = *reinterpret_cast<const uint4*>(x + (16 * wn + 8 * j + g) * kSPitch + col);
        mma_16816<true>(acc[j], Ag.x, Ag8.x, Ag.y, Ag8.y, B.x, B.y);
        mma_16816<true>(acc[j], Ag.z, Ag8.z, Ag.w, Ag8.w, B.z, B.w);
      }
    }
    __syncthreads();  // every warp is done with this buffer before it is refilled
  }
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int e = e_base + 16 * wm + g + ((r & 2) ? 8 : 0);
      const int t = t_base + 16 * wn + 8 * j + 2 * q + (r & 1);
      if (e < E && t < T) logits[static_cast<size_t>(t) * E + e] = acc[j][r];
    }
}

}  // namespace

cudaError_t launch_router(const uint16_t* X, int T, int d, const uint16_t* Wr, int E, float* logits,
                          cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  {
    const cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(router_smem_kernel), kSSmemBytes);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  timer_begin(kKRouter, stream);
  if (T <= kRowsMaxT) {
    cfg.gridDim = dim3((E + kRowsThreads / 32 - 1) / (kRowsThreads / 32));
    cfg.blockDim = dim3(kRowsThreads);
    e = cudaLaunchKernelEx(&cfg, router_rows_kernel, X, T, d, Wr, E, logits);
  } else {
    cfg.gridDim = dim3((E + kSE - 1) / kSE, (T + kST - 1) / kST);
    cfg.blockDim = dim3(kRouterThreads);
    cfg.dynamicSmemBytes = kSSmemBytes;
    e = cudaLaunchKernelEx(&cfg, router_smem_kernel, X, T, d, Wr, E, logits);
  }
  timer_end(kKRouter, stream);
  return e;
}

}  // namespace bm
