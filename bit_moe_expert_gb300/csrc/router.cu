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
// Three shapes.  Up to 32 tokens: a warp per router row on the CUDA cores, each
// lane with its whole share of the row in flight at once (the rows stream
// from HBM once; the products of bf16 values are exact in fp32, each sum is
// rounded once per step); a lane's partial sums are combined across the warp
// in a fixed tree.  More tokens: the tensor-core MMAs below on a CTA tile of 32
// experts x 64 tokens; the tiles of each 128-wide K chunk are staged in shared
// memory with cp.async, four chunks in flight, so every byte is read from L2
// once per CTA, and each warp multiplies 16 experts x 16 tokens from there.
// That shape is kept for router sizes the third one does not take.  More than
// 32 tokens, E a multiple of 128 and d of 256: the fifth-generation tensor
// cores.  A CTA multiplies 128 router rows (the MMA's M, one per TMEM lane) by
// 64 tokens (N, TMEM columns) over a quarter of K; both operands arrive by TMA
// in 128-byte-swizzled 64-wide K slices through a four-stage ring (the first
// four slices of router rows are requested before the previous kernel ends).
// The four CTAs of a thread-block cluster hold the four quarters: each drains
// its fp32 partial sums from TMEM into its shared memory (over the stages,
// which the MMAs are done with), and after a cluster barrier CTA r reads the
// four partials of tokens 16r .. 16r+15 through distributed shared memory and
// adds them in rank order, so the result does not depend on timing and needs
// no workspace.  97 KB of shared memory: two CTAs share an SM, one's loads
// overlapping the other's reduction.
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

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b, float acc) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc = fmaf(__uint_as_float(av[j] << 16), __uint_as_float(bv[j] << 16), acc);
    acc = fmaf(__uint_as_float(av[j] & 0xFFFF0000u), __uint_as_float(bv[j] & 0xFFFF0000u), acc);
  }
  return acc;
}

// kG tokens have their loads in flight together: 4 in general, 1 for the
// decode token (fewer registers, so that the CTAs fit beside a decode
// kernel's and can start while it finishes).
template <int kG>
__global__ void __launch_bounds__(kRowsThreads)
    router_rows_kernel(const uint16_t* __restrict__ X, int T, int d, const uint16_t* __restrict__ Wr, int E,
                       float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * (kRowsThreads / 32) + (threadIdx.x >> 5);
  const bool live = e < E;
  const int n16 = d / 8;  // 16-byte pieces per row
  const uint4* w = reinterpret_cast<const uint4*>(Wr + static_cast<size_t>(live ? e : 0) * d);
  const uint4* xr = reinterpret_cast<const uint4*>(X);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  // the router row does not come from the previous kernel: when it fits one
  // round (d <= 2048) it is loaded before waiting for that kernel and kept
  // in registers for every token
  const bool one_round = n16 <= 32 * kRowsU;
  uint4 w0[kRowsU];
#pragma unroll
  for (int u = 0; u < kRowsU; ++u)
    w0[u] = (one_round && live && lane + 32 * u < n16) ? __ldg(w + lane + 32 * u) : zero;
  pdl_wait();  // X may come from the previous kernel on the stream
  pdl_launch_dependents();
  if (!live) return;
  // tokens in groups of kG, every load of a group in flight together (longer
  // rows: the router row comes from HBM for the first group and from L1 after)
  for (int t0 = 0; t0 < T; t0 += kG) {
    float acc[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) acc[j] = 0.0f;
    if (one_round) {
      uint4 xv[kG][kRowsU];
#pragma unroll
      for (int u = 0; u < kRowsU; ++u) {
        const bool in = lane + 32 * u < n16;
#pragma unroll
        for (int j = 0; j < kG; ++j)
          xv[j][u] = (in && t0 + j < T) ? __ldg(xr + static_cast<size_t>(t0 + j) * n16 + lane + 32 * u) : zero;
      }
#pragma unroll
      for (int j = 0; j < kG; ++j)
#pragma unroll
        for (int u = 0; u < kRowsU; ++u) acc[j] = dot8_bf16(w0[u], xv[j][u], acc[j]);
    } else {
      for (int i0 = lane; i0 < n16; i0 += 32 * kRowsU) {
        uint4 wv[kRowsU], xv[kG][kRowsU];
#pragma unroll
        for (int u = 0; u < kRowsU; ++u) {
          const bool in = i0 + 32 * u < n16;
          wv[u] = in ? __ldg(w + i0 + 32 * u) : zero;
#pragma unroll
          for (int j = 0; j < kG; ++j)
            xv[j][u] = (in && t0 + j < T) ? __ldg(xr + static_cast<size_t>(t0 + j) * n16 + i0 + 32 * u) : zero;
        }
#pragma unroll
        for (int j = 0; j < kG; ++j)
#pragma unroll
          for (int u = 0; u < kRowsU; ++u) acc[j] = dot8_bf16(wv[u], xv[j][u], acc[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kG; ++j) {
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

// ---------------------------------------------------------------- tensor cores
constexpr int kTcK = 64;  // K per stage: one 128-byte swizzled row of each operand
constexpr int kTcStages = 4;
constexpr int kTcABytes = kRouterTcE * kTcK * 2;   // router rows of a stage
constexpr int kTcBBytes = kRouterTcT * kTcK * 2;   // token rows of a stage
constexpr int kTcStageBytes = kTcABytes + kTcBBytes;
constexpr int kTcThreads = 192;                    // warp 0 TMA, warp 1 MMA, warps 2-5 TMEM drain and sums
constexpr int kTcTmemCols = 64;                    // one fp32 column per token
constexpr int kTcSlice = kRouterTcT / kRouterTcSplit;          // tokens each CTA of the cluster sums
constexpr int kTcPartBytes = kRouterTcT * kRouterTcE * 4;       // this CTA's partial sums [token][router row], over the stages
constexpr int kTcRedVecs = kTcSlice * kRouterTcE / 4;           // float4 of a slice
constexpr int kTcRedIters = (kTcRedVecs + kTcThreads - 1) / kTcThreads;
constexpr int kTcSmemBytes = 1024 /*align*/ + kTcStages * kTcStageBytes + 256 /*barriers*/;
static_assert(kTcABytes % 1024 == 0 && kTcStageBytes % 1024 == 0, "stages keep the swizzle atoms aligned");
static_assert(kTcPartBytes <= kTcStages * kTcStageBytes, "the partial sums fit over the stages");
static_assert(2 * kTcSmemBytes <= 232448, "two CTAs per SM");
static_assert(kRouterTcE == 128 && kRouterTcT % 16 == 0 && kRouterTcT <= 256, "a valid M = 128 MMA shape");
static_assert(kRouterTcT % (4 * kRouterTcSplit) == 0, "whole float4 slices");

__global__ void __launch_bounds__(kTcThreads, 2)
    router_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap, int T,
                     int d, int E, float* __restrict__ logits) {
  extern __shared__ uint8_t s_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  // written only once every MMA has completed (acc_full), when every stage's
  // copies have landed and been read
  float* part = reinterpret_cast<float*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTcStages * kTcStageBytes);
  uint64_t* empty = full + kTcStages;
  uint64_t* acc_full = empty + kTcStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // the K quarter; the cluster spans gridDim.x
  const int t_base = blockIdx.y * kRouterTcT, e_base = blockIdx.z * kRouterTcE;
  const int kq = d / kRouterTcSplit;
  const int k0 = static_cast<int>(rank) * kq;
  const int nk = kq / kTcK;
  const int pre = nk < kTcStages ? nk : kTcStages;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], 1);   // the producer's expect_tx arrival; the bytes complete the phase
      mbar_init(&empty[i], 1);  // the MMA issuer's commit
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // the router rows do not come from the previous kernel: the first ring's
    // worth is requested at once, the tokens once it has finished (while warp
    // 1 allocates TMEM)
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
    for (int ks = 0; ks < pre; ++ks) {
      mbar_arrive_expect_tx(&full[ks], kTcStageBytes);
      tma_load_2d(stages + ks * kTcStageBytes, &wmap, &full[ks], k0 + ks * kTcK, e_base);
    }
    pdl_wait();  // X may come from the previous kernel
    for (int ks = 0; ks < pre; ++ks)
      tma_load_2d(stages + ks * kTcStageBytes + kTcABytes, &xmap, &full[ks], k0 + ks * kTcK, t_base);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool failed = false;
  uint32_t v[kRouterTcT];
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {  // the thread that issued the first copies
      int issued = pre;
      for (int ks = pre; ks < nk; ++ks) {
        const int st = ks % kTcStages;
        if (!mbar_wait(&empty[st], ((ks / kTcStages) - 1) & 1, abort_flag)) {
          failed = true;
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[st], kTcStageBytes);
        tma_load_2d(stages + st * kTcStageBytes, &wmap, &full[st], k0 + ks * kTcK, e_base);
        tma_load_2d(stages + st * kTcStageBytes + kTcABytes, &xmap, &full[st], k0 + ks * kTcK, t_base);
        issued = ks + 1;
      }
      // copies still in flight land before the CTA may exit
      for (int ks = issued > kTcStages ? issued - kTcStages : 0; ks < issued; ++ks)
        mbar_wait(&full[ks % kTcStages], (ks / kTcStages) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // shared-memory addresses stay below 2^18, so the descriptors' 14-bit
    // address field never carries into its neighbours; the four K = 16
    // slices of a stage are 32 bytes apart in the swizzled rows (2 in the
    // address field)
    const uint32_t idesc = idesc_bf16_f32(kRouterTcE, kRouterTcT);
    const uint64_t desc0 = smem_desc_sw128_kmajor(smem_u32(stages));
    for (int ks = 0; ks < nk; ++ks) {
      const int st = ks % kTcStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (ks / kTcStages) & 1, abort_flag))) {
        failed = true;
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      if (elect_one()) {
        const uint64_t a = desc0 + static_cast<uint64_t>((st * kTcStageBytes) >> 4);
        const uint64_t b = a + static_cast<uint64_t>(kTcABytes >> 4);
#pragma unroll
        for (int kk = 0; kk < kTcK / 16; ++kk) tc_mma_ss(tmem, a + 2 * kk, b + 2 * kk, idesc, (ks | kk) ? 1u : 0u);
        tc_commit(&empty[st]);
      }
      __syncwarp();
    }
    // arrives once every MMA issued above has completed (at once if none was)
    if (elect_one()) tc_commit(acc_full);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ TMEM drain
    // warp w may read TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31: its router rows
    if (__all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag))) {
      tc_fence_after();
      const uint32_t ta = tmem + ((32u * static_cast<uint32_t>(warp & 3)) << 16);
#pragma unroll
      for (int c = 0; c < kRouterTcT; c += 16) tmem_ld16(ta + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
      tc_wait_ld();
    } else {
      failed = true;
    }
  }
  // a wait that gave up anywhere turns this CTA's partial sums into NaN, so
  // the tiles' logits are NaN (which the routing kernel reports)
  const bool bad = __syncthreads_or(failed) != 0;
  if (warp >= 2) {
    const int row = 32 * (warp & 3) + lane;
#pragma unroll
    for (int t = 0; t < kRouterTcT; ++t) part[t * kRouterTcE + row] = bad ? __int_as_float(0x7fc00000) : __uint_as_float(v[t]);
  }
  tc_fence_before();
  cluster_arrive_release();  // every CTA's partial sums are in its shared memory
  cluster_wait();
  // the next kernel may start once this CTA's loads are done (not before, so
  // its CTAs do not compete with them; and after the TMEM allocation, so they
  // cannot hold the TMEM this CTA waits for)
  pdl_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    mbar_wait(acc_full, 0, nullptr);  // the MMAs are done with TMEM (already so unless a wait gave up)
    tmem_dealloc(tmem, kTcTmemCols);
  }

  // tokens kTcSlice * rank .. + kTcSlice - 1 of the tile: the four quarters'
  // partial sums added in rank order, read through distributed shared memory
  pdl_wait();  // the previous kernel may still read the logits written below
  {
    const uint32_t base = static_cast<uint32_t>(kTcSlice * static_cast<int>(rank) * kRouterTcE * 4);
    uint32_t src[kRouterTcSplit];
#pragma unroll
    for (int r = 0; r < kRouterTcSplit; ++r) src[r] = mapa_shared(part, static_cast<uint32_t>(r)) + base;
    const float* mine = part + kTcSlice * static_cast<int>(rank) * kRouterTcE;
    float4 p[kTcRedIters][kRouterTcSplit];
#pragma unroll
    for (int it = 0; it < kTcRedIters; ++it) {
      const int i = threadIdx.x + it * kTcThreads;
#pragma unroll
      for (int r = 0; r < kRouterTcSplit; ++r)
        if (i < kTcRedVecs)
          p[it][r] = r == static_cast<int>(rank) ? reinterpret_cast<const float4*>(mine)[i]
                                                 : ld_shared_cluster_f4(src[r] + 16u * static_cast<uint32_t>(i));
    }
#pragma unroll
    for (int it = 0; it < kTcRedIters; ++it) {
      const int i = threadIdx.x + it * kTcThreads;
      if (i >= kTcRedVecs) continue;
      float4 acc = p[it][0];
#pragma unroll
      for (int r = 1; r < kRouterTcSplit; ++r) {
        acc.x += p[it][r].x;
        acc.y += p[it][r].y;
        acc.z += p[it][r].z;
        acc.w += p[it][r].w;
      }
      const int t = t_base + kTcSlice * static_cast<int>(rank) + i / (kRouterTcE / 4);
      const int e = e_base + 4 * (i % (kRouterTcE / 4));
      if (t < T) *reinterpret_cast<float4*>(logits + static_cast<size_t>(t) * E + e) = acc;
    }
  }
  // no CTA leaves while another still reads its partial sums (the loads above
  // have returned: their values are stored)
  cluster_arrive_relaxed();
  cluster_wait();
}

}  // namespace

bool router_tc_shape(int T, int d, int E) {
  return T > kRowsMaxT && E % kRouterTcE == 0 && d % (kTcK * kRouterTcSplit) == 0 &&
         (T + kRouterTcT - 1) / kRouterTcT <= 65535 && E / kRouterTcE <= 65535;
}

cudaError_t launch_router(const uint16_t* X, int T, int d, const uint16_t* Wr, int E, float* logits,
                          const RouterMaps* maps, cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  if (maps && router_tc_shape(T, d, E)) {
    const cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(router_tc_kernel), kTcSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = kRouterTcSplit;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(kRouterTcSplit, (T + kRouterTcT - 1) / kRouterTcT, E / kRouterTcE);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmemBytes;
    timer_begin(kKRouter, stream);
    const cudaError_t le = cudaLaunchKernelEx(&cfg, router_tc_kernel, maps->x, maps->wr, T, d, E, logits);
    timer_end(kKRouter, stream);
    return le;
  }
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
    e = T == 1 ? cudaLaunchKernelEx(&cfg, router_rows_kernel<1>, X, T, d, Wr, E, logits)
               : cudaLaunchKernelEx(&cfg, router_rows_kernel<4>, X, T, d, Wr, E, logits);
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
