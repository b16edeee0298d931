// GPU-resident routing in one launch: top-k, histogram, exclusive scan, stable
// scatter and tile block map, with no host round trip ("Perplexity's Lily
// Beats MLX-LM on MacBook M5", section "Prefill: keep routing on the GPU,
// dequantize in flight": histogram, prefix scan, scatter and block map after
// every top-8 selection, kept inside one GPU submission).
//
// Each routing CTA takes a chunk of 32 tokens (one warp per token at a time)
// and selects their top k.  It then writes its
// per-expert counts and, for every assignment, the rank among the chunk's
// assignments to the same expert (computed in assignment order, so the result
// is stable).  The last CTA to finish (an atomic ticket, no spin wait) reduces
// the chunk counts into counts/offsets, turns them into per-chunk bases, places
// every assignment, and writes the block map.
//
// The routing weights (a softmax in fp64, which is slow on this GPU) are not on
// that chain: extra CTAs after the routing CTAs select the top k of 8 tokens
// each again (the same function, so the same selection) and write only the
// weights; they wait for nothing, so they run beside the routing CTAs.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace bm {

namespace {

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kBasesSmemLimit = 96 * 1024;  // per-chunk bases kept in shared memory up to this size
// Tokens per weight CTA (one per warp; the CTA's other warps leave at once).
// fp64 is slow on this GPU and shared by an SM's warps: 8 tokens per CTA
// instead of 16 spread the weights over twice the SMs (the 1024-token chunk's
// weight CTAs finished at 8.9 us, after the routing CTAs; the long-prefill
// step went from 0.467 to 0.452 ms).
constexpr int kWeightTokensPerCta = 8;
static_assert(kWeightTokensPerCta <= kRouteWarps, "a weight CTA's tokens fit its warps");

constexpr int kRouteMaxDevices = 64;
struct RouteSetup {
  bool done;
  int resident8, resident32;  // CTAs of route_kernel<8>, <32> resident at once (no dynamic shared memory)
};
RouteSetup g_route_setup[kRouteMaxDevices] = {};
std::mutex g_route_setup_mu;

// kPL: logits per lane (E <= 32 * kPL).
template <int kPL>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const float* __restrict__ logits, int T, int E,
                                                              int k, int block_rows, RouteOut out,
                                                              WsHeader* hdr, uint32_t* status,
                                                              int32_t* __restrict__ chunk_hist,
                                                              int32_t* __restrict__ local_rank, int bases_in_smem,
                                                              int gridsync, int nroute) {
  extern __shared__ int32_t s_bases[];  // [nchunks][E] exclusive per-chunk bases (last CTA, when they fit)
  __shared__ int32_t s_ids[kRouteTokensPerCta * kMaxK];
  __shared__ int32_t s_rank[kRouteTokensPerCta * kMaxK];
  __shared__ int32_t s_cnt[kMaxE];
  __shared__ uint32_t s_mask[kMaxE];  // tokens of the chunk (bit = token within the chunk) that chose expert e
  __shared__ int32_t s_off[kMaxE + 1];
  __shared__ int32_t s_boff[kMaxE + 1];
  __shared__ int32_t s_part[2][kRouteThreads];
  __shared__ int32_t s_base[kMaxE];  // grid-synchronised mode: this chunk's base within each expert
  __shared__ int s_is_last;

  pdl_wait();  // the previous kernel on the stream may still own our outputs
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int chunk = blockIdx.x;
  const int nchunks = nroute;
  const int t0 = chunk * kRouteTokensPerCta;
  const int ntok = max(0, min(kRouteTokensPerCta, T - t0));
  const int A = T * k;

  if (chunk >= nroute) {
    // ---- a weight CTA: one token per warp; the softmax over the selected
    // logits in fp64, summed in selection order, rounded once
    const int t = (chunk - nroute) * kWeightTokensPerCta + warp;
    if (warp < kWeightTokensPerCta && t < T) {
      int sel_i;
      float sel_v;
      bool finite;
      warp_topk_select<kPL>(logits + static_cast<size_t>(t) * E, E, k, lane, sel_i, sel_v, finite);
      const float wj = warp_topk_weights(sel_v, k, lane);
      if (lane < k) out.w[static_cast<size_t>(t) * k + lane] = wj;
    }
    return;
  }

  for (int e = threadIdx.x; e < E; e += kRouteThreads) s_mask[e] = 0u;
  __syncthreads();

  // ---- top-k, one warp per token
  static_assert(kRouteTokensPerCta <= 32, "a chunk's tokens are the bits of one word");
  auto publish = [&](int tl, int sel_i, bool finite) {
    if (!finite && lane == 0) record_status(status, MOE_ERR_NONFINITE);
    if (lane < k) {
      out.ids[static_cast<size_t>(t0 + tl) * k + lane] = sel_i;
      s_ids[tl * k + lane] = sel_i;
      atomicOr(&s_mask[sel_i], 1u << tl);
    }
  };
  if constexpr (kPL == 8) {
    // both of a warp's rows are in flight before either is selected
    static_assert(kRouteTokensPerCta == 2 * kRouteWarps, "two tokens per warp");
    float xv[2][8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int tl = warp + u * kRouteWarps;
      if (tl < ntok) topk_load_row8(logits + static_cast<size_t>(t0 + tl) * E, E, lane, xv[u]);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int tl = warp + u * kRouteWarps;
      if (tl < ntok) {
        int sel_i;
        float sel_v;
        bool finite;
        warp_topk_select_sorted_vals(xv[u], E, k, lane, sel_i, sel_v, finite);
        publish(tl, sel_i, finite);
      }
    }
  } else {
    for (int tl = warp; tl < ntok; tl += kRouteWarps) {
      int sel_i;
      float sel_v;
      bool finite;
      warp_topk_select<kPL>(logits + static_cast<size_t>(t0 + tl) * E, E, k, lane, sel_i, sel_v, finite);
      publish(tl, sel_i, finite);
    }
  }
  __syncthreads();

  // ---- stable per-chunk ranks: a token picks an expert at most once, so the
  // rank of assignment (token tl, slot j) among the chunk's assignments to
  // expert e, in assignment order, is the number of earlier tokens of the
  // chunk that chose e
  const int na = ntok * k;
  for (int a = threadIdx.x; a < na; a += kRouteThreads) {
    const int tl = a / k;
    s_rank[a] = __popc(s_mask[s_ids[a]] & ((1u << tl) - 1u));
  }
  for (int e = threadIdx.x; e < E; e += kRouteThreads) s_cnt[e] = __popc(s_mask[e]);
  __syncthreads();

  if (nchunks > 1 && gridsync) {
    // Every CTA is resident (the launch is sized for it): publish this chunk's
    // counts, wait for every chunk (bounded spin), then each CTA derives the
    // totals and its own chunk's bases and places its own assignments.
    for (int e = threadIdx.x; e < E; e += kRouteThreads) chunk_hist[static_cast<size_t>(chunk) * E + e] = s_cnt[e];
    __syncthreads();
    if (threadIdx.x == 0) {
      atom_add_acq_rel_gpu(&hdr->ticket, 1u);
      const long long tw = clock64();
      while (ld_acquire_gpu(&hdr->ticket) < static_cast<uint32_t>(nchunks)) {
        if (clock64() - tw > kWaitLimitCycles) {
          record_status(status, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
      int run = 0, mine = 0;
      for (int c0 = 0; c0 < nchunks; c0 += 32) {  // 32 loads in flight per round trip
        int h[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          h[i] = (c0 + i < nchunks) ? __ldcg(chunk_hist + static_cast<size_t>(c0 + i) * E + e) : 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (c0 + i == chunk) mine = run;
          run += h[i];
        }
      }
      s_cnt[e] = run;
      s_base[e] = mine;
    }
    __syncthreads();
  } else if (nchunks > 1) {
    // publish this chunk's counts and ranks, then the last CTA finishes
    for (int e = threadIdx.x; e < E; e += kRouteThreads) chunk_hist[static_cast<size_t>(chunk) * E + e] = s_cnt[e];
    for (int a = threadIdx.x; a < na; a += kRouteThreads) local_rank[static_cast<size_t>(t0) * k + a] = s_rank[a];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned ticket = atomicAdd(&hdr->ticket, 1u);
      s_is_last = (ticket == static_cast<unsigned>(nchunks - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    // counts and exclusive per-chunk bases; loads batched so they overlap
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
      int run = 0;
      for (int c0 = 0; c0 < nchunks; c0 += 8) {
        int h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          h[i] = (c0 + i < nchunks) ? __ldcg(chunk_hist + static_cast<size_t>(c0 + i) * E + e) : 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (c0 + i < nchunks) {
            if (bases_in_smem)
              s_bases[(c0 + i) * E + e] = run;
            else
              chunk_hist[static_cast<size_t>(c0 + i) * E + e] = run;
          }
          run += h[i];
        }
      }
      s_cnt[e] = run;
    }
    __syncthreads();
  }
  const bool writer = !gridsync || chunk == 0;  // in grid-synchronised mode CTA 0 writes the per-expert outputs
  if (writer)
    for (int e = threadIdx.x; e < E; e += kRouteThreads) out.counts[e] = s_cnt[e];

  // ---- exclusive scans over experts: row offsets and tile offsets
  {
    const int per = (E + kRouteThreads - 1) / kRouteThreads;
    const int lo = threadIdx.x * per;
    const int hi = min(E, lo + per);
    int rs = 0, bs = 0;
    for (int e = lo; e < hi; ++e) {
      rs += s_cnt[e];
      bs += (s_cnt[e] + block_rows - 1) / block_rows;
    }
    // warp-level inclusive scans of the per-thread sums, then across warps
    int ir = rs, ib = bs;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int r2 = __shfl_up_sync(0xffffffffu, ir, off);
      const int b2 = __shfl_up_sync(0xffffffffu, ib, off);
      if (lane >= off) {
        ir += r2;
        ib += b2;
      }
    }
    if (lane == 31) {
      s_part[0][warp] = ir;
      s_part[1][warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
      int wr = lane < kRouteWarps ? s_part[0][lane] : 0;
      int wb = lane < kRouteWarps ? s_part[1][lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int r2 = __shfl_up_sync(0xffffffffu, wr, off);
        const int b2 = __shfl_up_sync(0xffffffffu, wb, off);
        if (lane >= off) {
          wr += r2;
          wb += b2;
        }
      }
      if (lane < kRouteWarps) {
        s_part[0][kRouteWarps + lane] = wr;  // inclusive totals per warp
        s_part[1][kRouteWarps + lane] = wb;
      }
    }
    __syncthreads();
    const int wbase_r = warp > 0 ? s_part[0][kRouteWarps + warp - 1] : 0;
    const int wbase_b = warp > 0 ? s_part[1][kRouteWarps + warp - 1] : 0;
    rs = wbase_r + ir - rs;  // exclusive prefix of this thread's slice
    bs = wbase_b + ib - bs;
    for (int e = lo; e < hi; ++e) {
      s_off[e] = rs;
      s_boff[e] = bs;
      rs += s_cnt[e];
      bs += (s_cnt[e] + block_rows - 1) / block_rows;
    }
    if (threadIdx.x == kRouteThreads - 1) {
      s_off[E] = s_part[0][2 * kRouteWarps - 1];
      s_boff[E] = s_part[1][2 * kRouteWarps - 1];
    }
  }
  __syncthreads();
  if (writer) {
    for (int e = threadIdx.x; e <= E; e += kRouteThreads) out.offsets[e] = s_off[e];
    if (threadIdx.x == 0) *out.num_blocks = s_boff[E];

    // ---- block map
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
      const int cnt = s_cnt[e];
      int b = s_boff[e];
      for (int r = 0; r < cnt; r += block_rows, ++b) {
        out.block_map[3 * b + 0] = e;
        out.block_map[3 * b + 1] = s_off[e] + r;
        out.block_map[3 * b + 2] = min(block_rows, cnt - r);
      }
    }
  }

  // ---- scatter: position = offsets[e] + base of the chunk for e + rank within the chunk
  if (nchunks > 1 && gridsync) {
    for (int a = threadIdx.x; a < na; a += kRouteThreads) {
      const int e = s_ids[a];
      const int pos = s_off[e] + s_base[e] + s_rank[a];
      const int ga = t0 * k + a;
      out.perm[pos] = ga;
      out.inv_perm[ga] = pos;
    }
    __syncthreads();
    if (threadIdx.x == 0 && atom_add_acq_rel_gpu(&hdr->route_done, 1u) == static_cast<uint32_t>(nchunks - 1)) {
      // every CTA has passed the barrier: ready for the next call
      hdr->ticket = 0;
      hdr->route_done = 0;
      __threadfence();
    }
  } else if (nchunks == 1) {
    for (int a = threadIdx.x; a < na; a += kRouteThreads) {
      const int pos = s_off[s_ids[a]] + s_rank[a];
      out.perm[pos] = a;
      out.inv_perm[a] = pos;
    }
  } else {
    constexpr int kU = 8;
    for (int a0 = threadIdx.x; a0 < A; a0 += kRouteThreads * kU) {
      int e[kU], rk[kU];
#pragma unroll
      for (int i = 0; i < kU; ++i) {
        const int a = a0 + i * kRouteThreads;
        e[i] = a < A ? __ldcg(out.ids + a) : 0;
        rk[i] = a < A ? __ldcg(local_rank + a) : 0;
      }
#pragma unroll
      for (int i = 0; i < kU; ++i) {
        const int a = a0 + i * kRouteThreads;
        if (a < A) {
          const int c = (a / k) / kRouteTokensPerCta;
          const int base = bases_in_smem ? s_bases[c * E + e[i]]
                                         : __ldcg(chunk_hist + static_cast<size_t>(c) * E + e[i]);
          const int pos = s_off[e[i]] + base + rk[i];
          out.perm[pos] = a;
          out.inv_perm[a] = pos;
        }
      }
    }
    if (threadIdx.x == 0) hdr->ticket = 0;  // ready for the next call
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int block_rows, const RouteOut& out,
                         void* ws, cudaStream_t stream, bool pdl, uint32_t* status) {
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  if (!status) status = &hdr->status;
  const int nchunks = T > 0 ? (T + kRouteTokensPerCta - 1) / kRouteTokensPerCta : 1;
  int32_t* chunk_hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + sizeof(WsHeader));
  int32_t* local_rank = chunk_hist + route_hist_elems(T, E);
  const size_t bases_bytes = nchunks > 1 ? static_cast<size_t>(nchunks) * E * 4 : 0;
  const int bases_in_smem = (nchunks > 1 && bases_bytes <= static_cast<size_t>(kBasesSmemLimit)) ? 1 : 0;

  // One-time set-up per device (the dynamic shared-memory limit, and how many
  // CTAs of each instantiation fit at once), under a lock: host threads may
  // make their first calls on different devices at the same time.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kRouteMaxDevices) return cudaErrorInvalidDevice;
  int resident8 = 0, resident32 = 0;
  {
    std::lock_guard<std::mutex> lock(g_route_setup_mu);
    RouteSetup& su = g_route_setup[dev];
    if (!su.done) {
      cudaError_t e1 = cudaFuncSetAttribute(route_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBasesSmemLimit);
      if (e1 != cudaSuccess) return e1;
      cudaError_t e2 = cudaFuncSetAttribute(route_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBasesSmemLimit);
      if (e2 != cudaSuccess) return e2;
      int sms = 0, per8 = 0, per32 = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per8, route_kernel<8>, kRouteThreads, 0) == cudaSuccess &&
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per32, route_kernel<32>, kRouteThreads, 0) == cudaSuccess) {
        su.resident8 = sms * per8;
        su.resident32 = sms * per32;
      }
      su.done = true;
    }
    resident8 = su.resident8;
    resident32 = su.resident32;
  }
  // Grid-synchronised mode when every chunk's CTA can be resident at once
  // (leaving room for other work); otherwise the last CTA finishes alone.
  // MOE_ROUTE_MODE=ticket or =gridsync forces one of them (A/B and tests; a
  // forced grid-synchronised launch still needs every CTA resident, so it is
  // only taken when they fit).
  int gridsync = (nchunks > 1 && nchunks <= (E <= 256 ? resident8 : resident32) / 2) ? 1 : 0;
  if (const char* m = std::getenv("MOE_ROUTE_MODE")) {
    if (!std::strcmp(m, "ticket")) gridsync = 0;
    if (!std::strcmp(m, "gridsync") && nchunks > 1 && nchunks <= (E <= 256 ? resident8 : resident32)) gridsync = 1;
  }
  const int nweight = (T + kWeightTokensPerCta - 1) / kWeightTokensPerCta;  // weight CTAs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nchunks + nweight);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = (bases_in_smem && !gridsync) ? bases_bytes : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  timer_begin(kKRoute, stream);
  const cudaError_t err =
      E <= 256 ? cudaLaunchKernelEx(&cfg, route_kernel<8>, logits, T, E, k, block_rows, out, hdr, status,
                                    chunk_hist, local_rank, bases_in_smem && !gridsync, gridsync, nchunks)
               : cudaLaunchKernelEx(&cfg, route_kernel<32>, logits, T, E, k, block_rows, out, hdr, status,
                                    chunk_hist, local_rank, bases_in_smem && !gridsync, gridsync, nchunks);
  timer_end(kKRoute, stream);
  return err;
}

size_t route_hist_elems(int T, int E) {
  const int nchunks = T > 0 ? (T + kRouteTokensPerCta - 1) / kRouteTokensPerCta : 1;
  const size_t n = static_cast<size_t>(nchunks) * E;
  return (n + 63) & ~static_cast<size_t>(63);
}

// ------------------------------------------------------------------ prepack
namespace {
__global__ void prepack_kernel(const uint16_t* __restrict__ scale, const uint16_t* __restrict__ bias, int E,
                               int N, int G, uint32_t* __restrict__ sb) {
  // output index o = ((e*G + g)*N + n); input index i = ((e*N + n)*G + g)
  const size_t total = static_cast<size_t>(E) * G * N;
  for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < total;
       o += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(o % N);
    const size_t eg = o / N;
    const int g = static_cast<int>(eg % G);
    const int e = static_cast<int>(eg / G);
    const size_t i = (static_cast<size_t>(e) * N + n) * G + g;
    sb[o] = static_cast<uint32_t>(scale[i]) | (static_cast<uint32_t>(bias[i]) << 16);
  }
}

// Inside a word, codes k = 0..7 (k at bits 4k) are reordered so that code 2p
// sits at bits 4p and code 2p+1 at bits 4p+16: one mask then takes a pair of
// adjacent codes into the two halves of a 32-bit register.
__device__ __forceinline__ uint32_t interleave_nibbles(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int k = 2 * (i & 3) + (i >> 2);
    r |= ((w >> (4 * k)) & 0xFu) << (4 * i);
  }
  return r;
}
__device__ __forceinline__ uint4 interleave_nibbles(uint4 v) {
  return make_uint4(interleave_nibbles(v.x), interleave_nibbles(v.y), interleave_nibbles(v.z),
                    interleave_nibbles(v.w));
}

// codes [E][N][K/8] -> [E][K/64][N][8]: each row's 32-byte piece of one group
// moves next to the same group's piece of the next row; the codes of every
// word are interleaved (interleave_nibbles)
// 2-bit codes: inside a word, codes k = 0..15 (k at bits 2k) are reordered so
// that code 2p sits at bits 2p and code 2p+1 at bits 2p+16: one mask again
// takes a pair of adjacent codes into the two halves of a register.
__device__ __forceinline__ uint32_t interleave_pairs2(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int k = 2 * (i & 7) + (i >> 3);
    r |= ((w >> (2 * k)) & 0x3u) << (2 * i);
  }
  return r;
}
__device__ __forceinline__ uint4 interleave_pairs2(uint4 v) {
  return make_uint4(interleave_pairs2(v.x), interleave_pairs2(v.y), interleave_pairs2(v.z), interleave_pairs2(v.w));
}

// 3-bit codes: one row's 64 codes of a group (192 bits, code c at bits 3c of
// the six words) -> two planes in the same six words.  Words 0..3: the low
// two bits in the 2-bit interleaved order (word j = columns 16j .. 16j+15,
// column 16j+2p+h at bits 2p+16h).  Words 4, 5: the high bits, column
// 16j+2p+h at bit 16h + 8(j&1) + p of word 4 + j/2, so that the high bits of
// the code pair (2p, 2p+1) of 16-column block j sit p bits above bit 0 and
// bit 16 once the word is shifted right by 8(j&1).
__device__ __forceinline__ void repack3(const uint32_t (&in)[6], uint32_t (&out)[6]) {
#pragma unroll
  for (int i = 0; i < 6; ++i) out[i] = 0u;
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    const int bit = 3 * c, wi = bit >> 5, sh = bit & 31;
    uint32_t code = in[wi] >> sh;
    if (sh > 29) code |= in[wi + 1] << (32 - sh);
    code &= 7u;
    const int j = c >> 4, p = (c & 15) >> 1, h = c & 1;
    out[j] |= (code & 3u) << (2 * p + 16 * h);
    out[4 + (j >> 1)] |= (code >> 2) << (16 * h + 8 * (j & 1) + p);
  }
}

__global__ void prepack_codes3_kernel(const uint2* __restrict__ q, int E, int N, int G, uint2* __restrict__ qp) {
  const size_t total = static_cast<size_t>(E) * G * N;
  for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < total;
       o += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(o % N);
    const size_t eg = o / N;
    const int g = static_cast<int>(eg % G);
    const int e = static_cast<int>(eg / G);
    const size_t i = (static_cast<size_t>(e) * N + n) * G + g;  // the piece's 24 bytes: three 8-byte units
    uint32_t in[6], out[6];
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      const uint2 v = q[3 * i + u];
      in[2 * u] = v.x;
      in[2 * u + 1] = v.y;
    }
    repack3(in, out);
#pragma unroll
    for (int u = 0; u < 3; ++u) qp[3 * o + u] = make_uint2(out[2 * u], out[2 * u + 1]);
  }
}

// one row's piece of one group: 32 bytes (4-bit codes) or 16 bytes (2-bit)
template <int kBits>
__global__ void prepack_codes_kernel(const uint4* __restrict__ q, int E, int N, int G, uint4* __restrict__ qp) {
  constexpr int kU4 = kBits / 2;  // 16-byte units per piece
  const size_t total = static_cast<size_t>(E) * G * N;
  for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < total;
       o += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(o % N);
    const size_t eg = o / N;
    const int g = static_cast<int>(eg % G);
    const int e = static_cast<int>(eg / G);
    const size_t i = (static_cast<size_t>(e) * N + n) * G + g;
#pragma unroll
    for (int u = 0; u < kU4; ++u)
      qp[kU4 * o + u] = kBits == 4 ? interleave_nibbles(q[kU4 * i + u]) : interleave_pairs2(q[kU4 * i + u]);
  }
}
}  // namespace

// ------------------------------------------------------------------ dequantisation to fp16
namespace {
// W[e][n][k] = fp16(q * scale + bias) of one prepacked matrix: the weights a
// kernel without fused dequantisation would read.  One thread per 16 columns
// of one row and group: it reads the row's code words of the group and its
// (scale, bias) word and writes 32 bytes.  The code of column c of a group, in
// the prepacked order (see include/moe.h): 4-bit, word c/8, bits 4p + 16h with
// p = (c%8)/2, h = c%2; 2-bit, word c/16, bits 2p + 16h with p = (c%16)/2;
// 3-bit, those two bits from words 0..3 and the high bit at bit 16h + 8(j%2)
// + p of word 4 + j/2, j = c/16.
template <int kBits>
__device__ __forceinline__ uint32_t prepacked_code(const uint32_t* w, int c) {
  if constexpr (kBits == 4) return (w[c >> 3] >> (4 * ((c & 7) >> 1) + 16 * (c & 1))) & 0xFu;
  const int j = c >> 4, p = (c & 15) >> 1, h = c & 1;
  const uint32_t lo = (w[j] >> (2 * p + 16 * h)) & 0x3u;
  if constexpr (kBits == 2) return lo;
  return lo | (((w[4 + (j >> 1)] >> (16 * h + 8 * (j & 1) + p)) & 1u) << 2);
}

template <int kBits>
__global__ void dequant_kernel(const uint32_t* __restrict__ qp, const uint32_t* __restrict__ sb, int E, int N, int G,
                               uint16_t* __restrict__ W) {
  constexpr int kWpg = 2 * kBits;
  const size_t total = static_cast<size_t>(E) * G * N * 4;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int part = static_cast<int>(i & 3);  // columns 16 part .. 16 part + 15 of the group
    const size_t egn = i >> 2;                   // ((e * G + g) * N + n)
    const int n = static_cast<int>(egn % N);
    const size_t eg = egn / N;
    const int g = static_cast<int>(eg % G);
    const size_t e = eg / G;
    uint32_t w[kWpg];
#pragma unroll
    for (int u = 0; u < kWpg; ++u) w[u] = __ldg(qp + egn * kWpg + u);
    const uint32_t p = __ldg(sb + egn);
    const float scale = __uint_as_float(p << 16), bias = __uint_as_float(p & 0xFFFF0000u);
    uint32_t out[8];
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const float v0 = fmaf(static_cast<float>(prepacked_code<kBits>(w, 16 * part + c)), scale, bias);
      const float v1 = fmaf(static_cast<float>(prepacked_code<kBits>(w, 16 * part + c + 1)), scale, bias);
      out[c / 2] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v0))) |
                   (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v1))) << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(W + (e * N + n) * static_cast<size_t>(G) * 64 + g * 64 + 16 * part);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}
}  // namespace

cudaError_t launch_dequant(const uint32_t* qp, const uint32_t* sb, int E, int N, int K, int bits, uint16_t* W,
                           cudaStream_t stream) {
  const int G = K / 64;
  const size_t total = static_cast<size_t>(E) * G * N * 4;
  const int threads = 256;
  const size_t blocks = (total + threads - 1) / threads;
  const int grid = static_cast<int>(blocks < 65536 ? blocks : 65536);
  if (bits == 2)
    dequant_kernel<2><<<grid, threads, 0, stream>>>(qp, sb, E, N, G, W);
  else if (bits == 3)
    dequant_kernel<3><<<grid, threads, 0, stream>>>(qp, sb, E, N, G, W);
  else
    dequant_kernel<4><<<grid, threads, 0, stream>>>(qp, sb, E, N, G, W);
  return cudaGetLastError();
}

cudaError_t launch_prepack_codes(const uint32_t* q, int E, int N, int K, int bits, uint32_t* qp,
                                 cudaStream_t stream) {
  const int G = K / 64;
  const size_t total = static_cast<size_t>(E) * G * N;
  const int threads = 256;
  const size_t blocks = (total + threads - 1) / threads;
  const int grid = static_cast<int>(blocks < 65536 ? blocks : 65536);
  timer_begin(kKPrepack, stream);
  if (bits == 3)
    prepack_codes3_kernel<<<grid, threads, 0, stream>>>(reinterpret_cast<const uint2*>(q), E, N, G,
                                                        reinterpret_cast<uint2*>(qp));
  else if (bits == 2)
    prepack_codes_kernel<2><<<grid, threads, 0, stream>>>(reinterpret_cast<const uint4*>(q), E, N, G,
                                                          reinterpret_cast<uint4*>(qp));
  else
    prepack_codes_kernel<4><<<grid, threads, 0, stream>>>(reinterpret_cast<const uint4*>(q), E, N, G,
                                                          reinterpret_cast<uint4*>(qp));
  const cudaError_t err = cudaGetLastError();
  timer_end(kKPrepack, stream);
  return err;
}

cudaError_t launch_prepack(const uint16_t* scale, const uint16_t* bias, int E, int N, int K, uint32_t* sb,
                           cudaStream_t stream) {
  const int G = K / 64;
  const size_t total = static_cast<size_t>(E) * G * N;
  const int threads = 256;
  const size_t blocks = (total + threads - 1) / threads;
  const int grid = static_cast<int>(blocks < 65536 ? blocks : 65536);
  timer_begin(kKPrepack, stream);
  prepack_kernel<<<grid, threads, 0, stream>>>(scale, bias, E, N, G, sb);
  const cudaError_t err = cudaGetLastError();
  timer_end(kKPrepack, stream);
  return err;
}

}  // namespace bm

// ------------------------------------------------------------------ routing without a workspace
// The scratch of moe_route_noalloc: one file-scope device array, loaded with
// the module on every device that uses the library.  Host code must not pass
// the name itself to a kernel (on the host it is only a stand-in); the device
// address comes from cudaGetSymbolAddress, looked up with the device current.
// The address belongs to the CUDA context the module was loaded into: it is
// cached per device together with that context, and looked up again when the
// device's current context is a different one (after cudaDeviceReset).
namespace bm {
namespace {

static __device__ __align__(256) unsigned char g_route_scratch[MOE_ROUTE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
  void* ctx;   // the context the address was looked up in
  void* addr;  // device address of g_route_scratch in that context
};
ScratchAddr g_scratch[kMaxDevices] = {};

typedef int (*CtxGetCurrentFn)(void**);  // cuCtxGetCurrent: CUresult (CUcontext*)
CtxGetCurrentFn g_ctx_get = nullptr;
std::once_flag g_ctx_once;

// The current CUDA context of this thread (null if none or unavailable).
void* current_context() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
  });
  void* ctx = nullptr;
  if (!g_ctx_get || g_ctx_get(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of the scratch array on the current device (null on error).
// The first call in a context makes the runtime load the module there.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* ctx = current_context();  // null before the runtime has made the device's context current
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& sa = g_scratch[dev];
  if (!sa.addr || !ctx || sa.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return nullptr;
    sa.addr = p;
    sa.ctx = current_context();  // the context the runtime looked the address up in
  }
  return sa.addr;
}

}  // namespace
}  // namespace bm

extern "C" moe_status moe_route_noalloc(const float* logits, int T, int E, int k, int block_rows,
                                        moe_routing* out, moe_stream stream) {
  using namespace bm;
  if (!out || T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > kMaxK || k > E) return MOE_ERR_UNSUPPORTED;
  if (block_rows < 1 || block_rows > kMaxBlockRows) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * k > MOE_ROUTE_NOALLOC_MAX_ASSIGNMENTS ||
      route_hist_elems(T, E) > static_cast<size_t>(MOE_ROUTE_NOALLOC_MAX_HIST))
    return MOE_ERR_UNSUPPORTED;
  if (!out->counts || !out->offsets || !out->block_map || !out->num_blocks) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !out->ids || !out->w || !out->perm || !out->inv_perm)) return MOE_ERR_INVALID_ARG;

  void* scratch = scratch_address();
  if (!scratch) return MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The arrival counters must start at zero.  The status word (the header's
  // first word) is left alone: an error stays recorded until
  // moe_route_noalloc_check_status reads it.
  static_assert(offsetof(WsHeader, status) == 0, "status word first");
  if (cudaMemsetAsync(static_cast<char*>(scratch) + sizeof(uint32_t), 0, sizeof(WsHeader) - sizeof(uint32_t), st) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  out->block_rows = block_rows;
  RouteOut o{out->ids, out->w, out->counts, out->offsets, out->perm, out->inv_perm, out->block_map, out->num_blocks};
  if (launch_route(logits, T, E, k, block_rows, o, scratch, st, false) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" moe_status moe_route_noalloc_check_status(moe_stream stream) {
  using namespace bm;
  void* scratch = scratch_address();
  if (!scratch) return MOE_ERR_CUDA;
  return moe_check_status(scratch, stream);
}
