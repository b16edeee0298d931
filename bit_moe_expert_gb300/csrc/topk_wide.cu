// Exact top-K of each row of a wide score matrix ("Squeezing a 26B diffusion
// LLM onto a Mac", section "The optimizations that worked", item 1: the
// sampler needs only the top ~64 of 262,144 logits per position; a two-stage
// chunk-max selection finds them exactly).
//
// Order: a larger value first, a lower index first among equal values (-0.0
// equals +0.0).  Every entry gets the 64-bit key (monotone value key << 32 |
// ~index), so the order is total and every comparison below is strict.
//
// One CTA per row (persistent over rows; two CTAs per SM, so that one CTA's
// selection overlaps the other's streaming and 256 rows fit one wave), three
// phases:
//   1. stream the row once; each 256-entry chunk's largest value goes to
//      shared memory (a warp per chunk, eight chunks of loads in flight per
//      warp), as the chunk key (value key << 32 | ~chunk index);
//   2. select the K chunks ranked first by (largest value, lower chunk index):
//      a radix select (8 bits a pass) finds theta, the K-th largest chunk
//      maximum, and a prefix over the chunks equal to it takes the first ones;
//   3. re-read those chunks (L2), keep every entry whose value is at least
//      theta, rank the kept entries' keys (or sort them, when ties make them
//      many) and write the first K.  When ties make more candidates than the
//      buffer holds, a radix select over their 64-bit keys (8 bits a pass,
//      re-reading the chunks) finds the K-th largest key first, and only the K
//      keys at or above it are kept.
// Exactness.  Chunks are ranked by (largest value, lower chunk index).  Every
// chunk ranked above the chunk of an entry x holds an entry of larger key than
// x (a larger value, or the same value at a lower index, chunks being
// contiguous), so a top-K entry's chunk has fewer than K chunks above it and is
// selected.  The K selected maxima are K distinct entries of value at least
// theta, so every top-K entry has a value of at least theta.  Nothing is
// approximate; the candidates are a superset of the top K.
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace bm {

namespace {

constexpr int kWideThreads = 512;
constexpr int kWideWarps = kWideThreads / 32;
constexpr int kWideChunk = 256;  // entries per chunk: 8 per lane
constexpr int kWideU = 4;        // chunks of loads in flight per warp (64 KB per CTA, 128 KB per SM)
constexpr int kWideCand = 2048;  // candidate buffer (keys); more candidates take the radix-select path

__device__ __forceinline__ uint64_t wide_key(float v, int i) {
  return (static_cast<uint64_t>(topk_key(v)) << 32) | static_cast<uint32_t>(~i);
}

// Sorts n (a power of two) keys of shared memory into descending order; the
// whole CTA takes part and leaves synchronised.
__device__ void bitonic_desc(uint64_t* a, int n) {
  for (int k = 2; k <= n; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += kWideThreads) {
        const int lo = 2 * i - (i & (j - 1));  // the pair (lo, lo + j) of compare distance j
        const bool desc = (lo & k) == 0;       // direction of the bitonic run lo belongs to
        const uint64_t x = a[lo], y = a[lo + j];
        if ((x < y) == desc) {
          a[lo] = y;
          a[lo + j] = x;
        }
      }
      __syncthreads();
    }
}

// Lane `lane`'s 8 entries of chunk c (zero past V): two 16-byte loads when the
// row allows it, else scalar loads.
__device__ __forceinline__ void load_chunk8(const float* __restrict__ x, int V, int c, int lane, bool vec,
                                            float (&v)[8]) {
  const int base = c * kWideChunk + 8 * lane;
  if (vec) {
    // V % 4 == 0 and x 16-byte aligned: each float4 lies wholly inside or past the row
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 a = base < V ? __ldcs(reinterpret_cast<const float4*>(x + base)) : z;
    const float4 b = base + 4 < V ? __ldcs(reinterpret_cast<const float4*>(x + base + 4)) : z;
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = base + j < V ? __ldcs(x + base + j) : 0.0f;
  }
}

// Warp 0: the bin of s_hist (256 counts, scanned from the top bin down) that
// holds the take-th largest key; writes it to *bin and the count of the bins
// above it to *above.  The caller synchronises before and after.
__device__ __forceinline__ void find_bin(const int* s_hist, int take, int lane, int* bin, int* above) {
  int cnt[8], tot = 0;  // lane l owns bins 255 - 8l down to 248 - 8l
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    cnt[j] = s_hist[255 - 8 * lane - j];
    tot += cnt[j];
  }
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int p = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += p;
  }
  int acc = incl - tot;
  if (acc < take && take <= incl) {  // the bin holding the take-th largest key is this lane's
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (acc + cnt[j] >= take) {
        *bin = 255 - 8 * lane - j;
        *above = acc;
        break;
      }
      acc += cnt[j];
    }
  }
}

// Exclusive prefix over the CTA of one int per thread; returns the thread's
// prefix and, in *total, the sum.  Uses s_warp[kWideWarps] and synchronises.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int p = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += p;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWideWarps; ++w) {
    const int t = s_warp[w];
    before += w < warp ? t : 0;
    all += t;
  }
  __syncthreads();  // s_warp may be reused at once
  *total = all;
  return before + incl - v;
}

__global__ void __launch_bounds__(kWideThreads, 2)
    topk_wide_kernel(const float* __restrict__ logits, int T, int V, int K, int cand_cap, float* __restrict__ values,
                     int32_t* __restrict__ indices) {
  extern __shared__ uint64_t s_dyn[];  // candidates [cand_cap], then the chunk maxima' value keys
  __shared__ int s_hist[256];
  __shared__ int s_warp[kWideWarps];
  __shared__ int s_sel[64];
  __shared__ int s_n, s_nsel, s_bin, s_above;
  uint64_t* cand = s_dyn;
  uint32_t* ckv = reinterpret_cast<uint32_t*>(s_dyn + cand_cap);

  pdl_wait();  // the logits may come from the previous kernel on the stream
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nch = (V + kWideChunk - 1) / kWideChunk;
  for (int row = blockIdx.x; row < T; row += gridDim.x) {
    const float* x = logits + static_cast<size_t>(row) * V;
    const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15u) == 0);

    // ---- 1. chunk maxima (value keys)
    for (int c0 = warp * kWideU; c0 < nch; c0 += kWideWarps * kWideU) {
      float v[kWideU][8];
#pragma unroll
      for (int u = 0; u < kWideU; ++u) load_chunk8(x, c0 + u < nch ? V : 0, c0 + u, lane, vec, v[u]);
#pragma unroll
      for (int u = 0; u < kWideU; ++u) {
        const int base = (c0 + u) * kWideChunk + 8 * lane;
        uint32_t m = 0;  // below every value's key
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (base + j < V) m = max(m, topk_key(v[u][j]));
        m = __reduce_max_sync(0xffffffffu, m);
        if (lane == 0 && c0 + u < nch) ckv[c0 + u] = m;
      }
    }
    if (threadIdx.x == 0) {
      s_n = 0;
      s_nsel = 0;
    }
    __syncthreads();

    // ---- 2. the K chunks ranked first by (largest value, lower chunk index):
    // theta = the K-th largest chunk maximum (radix select, 8 bits a pass), then
    // every chunk above theta and the first `take` chunks equal to it
    uint32_t theta = 0;
    if (K >= nch) {
      for (int c = threadIdx.x; c < nch; c += kWideThreads) s_sel[c] = c;  // every chunk; every entry qualifies
      if (threadIdx.x == 0) s_nsel = nch;
    } else {
      uint32_t mask = 0;
      int take = K;  // chunks still to select at and below the current prefix
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kWideThreads) s_hist[i] = 0;
        __syncthreads();
        for (int c = threadIdx.x; c < nch; c += kWideThreads) {
          const uint32_t key = ckv[c];
          if ((key & mask) == theta) atomicAdd(&s_hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (warp == 0) find_bin(s_hist, take, lane, &s_bin, &s_above);
        __syncthreads();
        theta |= static_cast<uint32_t>(s_bin) << shift;
        mask |= 0xFFu << shift;
        take -= s_above;
      }
      // select: chunks above theta, and the first `take` chunks equal to it in chunk order
      constexpr int kMaxPer = (1 << 20) / kWideChunk / kWideThreads;  // chunks per thread at most
      const int per = (nch + kWideThreads - 1) / kWideThreads;
      const int c_lo = threadIdx.x * per;
      int ties = 0;
#pragma unroll
      for (int q = 0; q < kMaxPer; ++q)
        if (q < per && c_lo + q < nch) ties += ckv[c_lo + q] == theta ? 1 : 0;
      int total;
      int rank = block_exclusive_scan(ties, s_warp, &total);
#pragma unroll
      for (int q = 0; q < kMaxPer; ++q) {
        const int c = c_lo + q;
        if (q >= per || c >= nch) continue;
        const uint32_t key = ckv[c];
        bool pick = key > theta;
        if (key == theta) pick = rank++ < take;
        if (pick) s_sel[atomicAdd(&s_nsel, 1)] = c;
      }
    }
    __syncthreads();

    // ---- 3. candidates: the selected chunks' entries with values >= theta and
    // keys >= kappa (every load of a warp's chunks in flight together); fn(key)
    // sees each.  kappa is 0 except on the radix-select path.
    const int nsel = s_nsel;
    auto visit = [&](uint64_t kappa, auto&& fn) {
      constexpr int kPerWarp = 64 / kWideWarps;  // K <= 64 chunks over the warps
      float v[kPerWarp][8];
#pragma unroll
      for (int u = 0; u < kPerWarp; ++u) {
        const int sidx = warp + u * kWideWarps;
        load_chunk8(x, sidx < nsel ? V : 0, sidx < nsel ? s_sel[sidx] : 0, lane, vec, v[u]);
      }
#pragma unroll
      for (int u = 0; u < kPerWarp; ++u) {
        const int sidx = warp + u * kWideWarps;
        if (sidx >= nsel) continue;  // warp-uniform
        const int base = s_sel[sidx] * kWideChunk + 8 * lane;
        uint64_t keep[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const bool in = base + j < V && topk_key(v[u][j]) >= theta;
          keep[j] = in ? wide_key(v[u][j], base + j) : 0;
          if (keep[j] < kappa) keep[j] = 0;
        }
        fn(keep);
      }
    };
    // count and store (stores past the buffer are dropped; the count goes on)
    auto store = [&](const uint64_t (&keep)[8]) {
      int nk = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) nk += keep[j] != 0 ? 1 : 0;
      // warp-wide exclusive prefix of the lanes' counts, one shared atomic per warp
      int incl = nk;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int p = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += p;
      }
      int wbase = 0;
      if (lane == 31) wbase = atomicAdd(&s_n, incl);
      wbase = __shfl_sync(0xffffffffu, wbase, 31);
      int pos = wbase + incl - nk;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (keep[j] != 0) {
          if (pos < cand_cap) cand[pos] = keep[j];
          ++pos;
        }
    };
    visit(0ull, store);
    __syncthreads();
    if (s_n > cand_cap) {
      // More candidates than the buffer holds (ties with theta): kappa = the
      // K-th largest candidate key, by a radix select over the 64-bit keys,
      // then only the K keys >= kappa are stored (the keys are distinct).
      uint64_t kappa = 0, kmask = 0;
      int take = K;
      for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kWideThreads) s_hist[i] = 0;
        __syncthreads();
        visit(0ull, [&](const uint64_t (&keep)[8]) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (keep[j] != 0 && (keep[j] & kmask) == kappa) atomicAdd(&s_hist[(keep[j] >> shift) & 255u], 1);
        });
        __syncthreads();
        if (warp == 0) find_bin(s_hist, take, lane, &s_bin, &s_above);
        __syncthreads();
        kappa |= static_cast<uint64_t>(s_bin) << shift;
        kmask |= 0xFFull << shift;
        take -= s_above;
      }
      if (threadIdx.x == 0) s_n = 0;
      __syncthreads();
      visit(kappa, store);
      __syncthreads();
    }

    // ---- 4. order: the keys are distinct, so a key's rank is the number of
    // larger keys; few candidates (the usual case) are ranked directly, many
    // (heavy ties) are sorted
    const int n = s_n;  // at least K: the selected chunks' maxima (or all V >= K entries) qualify
    if (n <= 2 * kWideThreads) {
      for (int i = threadIdx.x; i < n; i += kWideThreads) {
        const uint64_t key = cand[i];
        int r = 0;
        for (int j = 0; j < n; ++j) r += cand[j] > key ? 1 : 0;
        if (r < K) {
          const int e = static_cast<int>(~static_cast<uint32_t>(key));
          indices[static_cast<size_t>(row) * K + r] = e;
          values[static_cast<size_t>(row) * K + r] = x[e];  // the entry itself (keeps the sign of a zero)
        }
      }
    } else {
      int p2 = 1;
      while (p2 < n) p2 <<= 1;
      for (int i = n + threadIdx.x; i < p2; i += kWideThreads) cand[i] = 0;
      __syncthreads();
      bitonic_desc(cand, p2);
      for (int j = threadIdx.x; j < K; j += kWideThreads) {
        const int e = static_cast<int>(~static_cast<uint32_t>(cand[j]));
        indices[static_cast<size_t>(row) * K + j] = e;
        values[static_cast<size_t>(row) * K + j] = x[e];
      }
    }
    __syncthreads();  // shared memory is reused by the next row
  }
}

}  // namespace

// candidates: a buffer of kWideCand keys (a power of two, for the sort); then
// one 4-byte value key per chunk
size_t topk_wide_smem_bytes(int V, int K) {
  (void)K;
  const int nch = (V + kWideChunk - 1) / kWideChunk;
  return static_cast<size_t>(kWideCand) * 8 + static_cast<size_t>(nch) * 4;
}

cudaError_t launch_topk_wide(const float* logits, int T, int V, int K, float* values, int32_t* indices,
                             int num_sms, cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  const size_t smem = topk_wide_smem_bytes(V, K);
  {
    const cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(topk_wide_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  int per_sm = 0;
  {
    const cudaError_t e =
        occupancy_per_sm(reinterpret_cast<const void*>(topk_wide_kernel), kWideThreads, smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
  }
  const int ctas = per_sm * num_sms;
  cfg.gridDim = dim3(static_cast<unsigned>(T < ctas ? T : ctas));
  cfg.blockDim = dim3(kWideThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  timer_begin(kKTopkWide, stream);
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, topk_wide_kernel, logits, T, V, K, kWideCand, values, indices);
  timer_end(kKTopkWide, stream);
  return e;
}

}  // namespace bm
