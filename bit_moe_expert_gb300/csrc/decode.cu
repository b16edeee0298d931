// Decode path (T <= 4 tokens).  "Perplexity's Lily Beats MLX-LM on MacBook
// M5", section "Prefill and decode are different problems": batch-1 decode is
// a matrix-vector product bound by memory bandwidth; section "Decode: minimize
// bytes per token": the expert input projections are fused with the gate
// activation and the output projection with the routing scores and the
// shared expert, and every weight byte is read once.
//
// Design (sm_103a): one launch per layer, one CTA per SM, two phases around
// one barrier over the grid.
//   phase 1  an item is 32 rows of the gate and up projections of one active
//            expert (the shared expert's items first).  CTA c takes items c,
//            c + grid, ...; it computes h = silu(x Wg^T) * (x Wu^T) for those
//            32 features of every token and writes it, in fp16, to the slot's
//            h record in global memory, with the sums of each 32 values.
//   barrier  every h record is complete.
//   phase 2  CTA c takes output rows [16c, 16c + 16) (and c + grid, ...): the
//            down projection of every active expert restricted to those rows,
//            times that expert's h and the token's routing weight, summed over
//            the experts, gives Y directly; nothing is reduced across CTAs.
// Every weight byte is loaded once, as soon as the routing is known (the
// shared expert's before the wait for the previous kernel).  One token (each
// CTA at most one item): the gate/up codes go straight from global memory
// into the MMA fragment registers of the warps that use them.  Otherwise TMA
// loads them into a ring of shared-memory stages (chunks of 8 groups of 64
// columns).  The phase-2 down rows (16 rows of one expert) come by TMA into a
// ring of their own and load while phase 1 runs.
//
// Arithmetic on the tensor cores (mma.sync m16n8k16, fp32 accumulators):
// weight rows are the 16 rows of the MMA, tokens its 8 columns (T <= 4 used).
// A code becomes 128 + q (bf16) or 1024 + q (fp16) with one mask (the codes of
// a word are interleaved: columns 2p and 2p+1 in bits 4p and 4p+16), and the
// affine map of each 64-column group is applied to the group's MMA result:
//   sum_k (q_k s + b) v_k = s * sum_k (M + q_k) v_k + (b - M s) * sum_k v_k.
// Phase 1 multiplies bf16 codes with the bf16 activations (exact products);
// phase 2 multiplies fp16 codes with fp16 h.
//
// The K order inside the MMA: lane (g, q) of a row holds the row's words 2q
// and 2q+1 of a group (an 8-byte load); step m of the group's four MMA steps
// takes code pairs 2(m&1) and 2(m&1)+1 of word 2q + (m>>1), which are columns
// 16q + 4m + {0,1} and + {2,3} of the group, so its activation operand is four
// consecutive values of the token (columns 16q .. 16q+15 over the four steps).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdlib>

#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace bm {

namespace {

constexpr int kWarps = 16;                   // compute warps
constexpr int kCons = kWarps * 32;           // compute threads
constexpr int kProducer = kWarps;            // the warp that issues every copy
constexpr int kThreads = kCons + 32;
constexpr int kRows1 = kDecodeRowsGU;           // gate/up rows per phase-1 item
constexpr int kChunk = kDecodeChunkGroups;      // groups per phase-1 stage
constexpr int kRows2 = kDecodeRowsDown;         // output rows per phase-2 block
constexpr int kS1 = 5;                          // phase-1 stages
constexpr int kSB1 = kS1;                       // phase-1 group-parameter buffers: one per stage
constexpr int kS2Max = 12;                      // phase-2 stages at most
constexpr int kMaxSlots = kMaxK * kGemvMaxT + 1;  // distinct experts of a call, plus the shared one
// kBits bits per weight code (4, 3 or 2): code words per row and 64-column group
template <int kBits>
constexpr int kWpg = 2 * kBits;
template <int kBits>
constexpr uint32_t kCodeQ = kChunk * kRows1 * 4 * kWpg<kBits>;  // bytes of one matrix's codes in a phase-1 stage
template <int kBits>
constexpr uint32_t kSt1 = 2 * kCodeQ<kBits>;  // phase-1 stage: gate codes, up codes
constexpr size_t kSmemMax = 227 * 1024;

static_assert(kWarps == 2 * kChunk, "phase 1 gives one warp to each (matrix, group) of a stage");
static_assert(kRows1 == 32 && kRows2 == 16, "fragment layout");
constexpr int kBars = 2 * kS1 + 3 * kS2Max + 3;  // mbarriers: full/empty per phase-1 stage, full (codes, h)/empty per
                                                 // phase-2 stage, x, routing weights, first h records
constexpr int kRegChunks = 4;  // phase-1 chunks held in registers (d <= 2048) when the codes are loaded directly

// Named barriers over the compute warps only (the producer may be waiting
// for room in the copy queue).
__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kCons) : "memory"); }
__device__ __forceinline__ void book_sync() { asm volatile("bar.sync 2, %0;" ::"r"(kCons) : "memory"); }

__host__ __device__ constexpr int div_up(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  int G1, nchunk, Imax, hs_stride, S2;
  size_t sb1;                 // bytes of one item's group parameters: gate [G1][32 rows], then up
  size_t hrec;                // bytes of one slot's h record: h fp16 [T][Imax], then half-group sums fp32 [T][hs_stride]
  size_t st2, st2_sb;         // phase-2 stage bytes (codes, then parameters); offset of the parameters
  size_t hring;               // h records of the phase-2 stages, [S2][hrec], consecutive like the global ones
  size_t ring1, sbuf1, xs, sx, red1, red2, wt, slot_e, rid, bk, misc, cnt, bars, ring2, total;
};

// TMA and bulk-copy destinations start on 128 bytes.
__host__ __device__ inline Layout layout(int T, int d, int I, int I_shared, int bits) {
  Layout L;
  L.G1 = d / 64;
  L.nchunk = div_up(L.G1, kChunk);
  L.Imax = I > I_shared ? I : I_shared;
  const int G2max = L.Imax / 64;
  L.hs_stride = static_cast<int>(round_up(L.Imax / 32, 4));
  L.hrec = static_cast<size_t>(T) * L.Imax * 2 + static_cast<size_t>(T) * L.hs_stride * 4;
  L.st2_sb = static_cast<size_t>(G2max) * kRows2 * 8 * bits;  // codes [G2][16 rows][2 bits words]
  L.st2 = round_up(L.st2_sb + static_cast<size_t>(G2max) * kRows2 * 4, 128);
  size_t o = 0;
  L.ring1 = o;
  o += static_cast<size_t>(kS1) * 2 * kChunk * kRows1 * 8 * bits;  // kSt1<bits>
  L.sb1 = round_up(2ull * L.G1 * kRows1 * 4, 128);
  L.sbuf1 = o;
  o += kSB1 * L.sb1;
  L.xs = o;  // x of every token, bf16 [T][d]
  o += round_up(static_cast<size_t>(T) * d * 2, 128);
  L.sx = o;  // sums of x over each group [T][G1]
  o += round_up(static_cast<size_t>(T) * L.G1 * 4, 16);
  L.red1 = o;  // phase-1 partial dots [warp][32 rows][T]
  o += static_cast<size_t>(kWarps) * kRows1 * T * 4;
  L.red2 = o;  // phase-2 partial rows [warp][16 rows][T]
  o += static_cast<size_t>(kWarps) * kRows2 * T * 4;
  L.wt = o;  // routing weight of each slot for each token [slot][T]
  o += static_cast<size_t>(kMaxSlots) * T * 4;
  L.slot_e = o;  // expert of each slot
  o += round_up(kMaxSlots * 4, 16);
  L.rid = o;  // the call's assignments: expert, weight, slot, selected logit [T*k] each; exp terms fp64 [T*k]
  o += 4ull * T * kMaxK * 4;
  o = round_up(o, 8);
  o += 8ull * T * kMaxK;
  L.bk = o;  // routing outputs' scratch: counts [E], offsets [E+1], tile offsets [E+1] (E <= 256)
  o += 3 * 260 * 4;
  L.misc = o;  // distinct routed experts
  o += 16;
  L.cnt = o;  // per-stage consumption counters; the job each phase-2 stage was last issued
  o += (kS1 + 2 * kS2Max) * 4;
  o = round_up(o, 8);
  L.bars = o;  // mbarriers
  o += static_cast<size_t>(kBars) * 8;
  o = round_up(o, 128);
  L.ring2 = o;
  const size_t room = kSmemMax > o + 128 ? kSmemMax - o - 128 : 0;
  size_t s2 = room / (L.st2 + L.hrec);
  if (s2 > kS2Max) s2 = kS2Max;
  L.S2 = static_cast<int>(s2);
  L.hring = o + s2 * L.st2;
  L.total = L.hring + s2 * L.hrec + 128;  // room to align the dynamic shared memory base
  return L;
}

// Four MMA steps over one 64-column group (see the K order above).
//   wa, wb: the codes of columns 16q .. 16q+15 of rows g and g+8 (4-bit
//   codes: words 2q, 2q+1; 2-bit codes: word q, in .x; 3-bit codes: the
//   low-bit word q in .x, the high-bit word shifted so that the pair
//   (2p, 2p+1)'s high bits sit at bits p and p+16, in .y); b: the activation
//   operand of the four steps (the same columns, token g).  Step m takes
//   columns 16q + 4m .. 16q + 4m + 3: two pairs of adjacent codes, each
//   formed by one mask from the interleaved word (3-bit codes: a second
//   mask adds the high bits as bit 2 of each half).
// x moved so that its bits P and P+16 land at bits 2 and 18 (P a constant
// once the caller's loop is unrolled)
__device__ __forceinline__ uint32_t shift_to_bit2(uint32_t x, int P) { return P < 2 ? x << (2 - P) : x >> (P - 2); }

template <bool kBF16, int kBits>
__device__ __forceinline__ void mma_group(uint2 wa, uint2 wb, const uint32_t (&b)[8], float (&dd)[4]) {
  constexpr uint32_t magic = kBF16 ? 0x43004300u : 0x64006400u;  // pairs (128, 128) / (1024, 1024)
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    uint32_t a0, a1, a2, a3;
    if constexpr (kBits == 4) {
      const uint32_t xa = m < 2 ? wa.x : wa.y;
      const uint32_t xb = m < 2 ? wb.x : wb.y;
      const int sh = (m & 1) * 8;
      a0 = lop3_and_or(xa >> sh, 0x000F000Fu, magic);
      a1 = lop3_and_or(xb >> sh, 0x000F000Fu, magic);
      a2 = lop3_and_or(xa >> (sh + 4), 0x000F000Fu, magic);
      a3 = lop3_and_or(xb >> (sh + 4), 0x000F000Fu, magic);
    } else {
      a0 = lop3_and_or(wa.x >> (4 * m), 0x00030003u, magic);  // code pair 2m
      a1 = lop3_and_or(wb.x >> (4 * m), 0x00030003u, magic);
      a2 = lop3_and_or(wa.x >> (4 * m + 2), 0x00030003u, magic);  // code pair 2m + 1
      a3 = lop3_and_or(wb.x >> (4 * m + 2), 0x00030003u, magic);
      if constexpr (kBits == 3) {  // high bits of pair P at bits P, P+16 -> bits 2, 18
        a0 = lop3_and_or(shift_to_bit2(wa.y, 2 * m), 0x00040004u, a0);
        a1 = lop3_and_or(shift_to_bit2(wb.y, 2 * m), 0x00040004u, a1);
        a2 = lop3_and_or(shift_to_bit2(wa.y, 2 * m + 1), 0x00040004u, a2);
        a3 = lop3_and_or(shift_to_bit2(wb.y, 2 * m + 1), 0x00040004u, a3);
      }
    }
    mma_16816<kBF16>(dd, a0, a1, a2, a3, b[2 * m], b[2 * m + 1]);
  }
}

// The codes of columns 16q .. 16q+15 of one row: 4-bit codes, two words;
// 2-bit codes, one word (in .x); 3-bit codes, low-bit word q and high-bit
// word 4 + q/2 shifted down by 8(q&1).
template <int kBits>
__device__ __forceinline__ uint2 load_codes(const uint32_t* row, int q) {
  if constexpr (kBits == 4) return *reinterpret_cast<const uint2*>(row + 2 * q);
  if constexpr (kBits == 3) return make_uint2(row[q], row[4 + (q >> 1)] >> (8 * (q & 1)));
  return make_uint2(row[q], 0u);
}

// The same code words read straight from global memory into registers (the
// 3-bit high-bit word unshifted: codes_fix shifts it where it is used, so the
// load is not waited for where it is issued).
template <int kBits>
__device__ __forceinline__ uint2 ldg_codes(const uint32_t* row, int q) {
  if constexpr (kBits == 4) return ldg_stream_v2(row + 2 * q);
  if constexpr (kBits == 3) return make_uint2(ldg_stream_u32(row + q), ldg_stream_u32(row + 4 + (q >> 1)));
  return make_uint2(ldg_stream_u32(row + q), 0u);
}
template <int kBits>
__device__ __forceinline__ uint2 codes_fix(uint2 w, int q) {
  if constexpr (kBits == 3) w.y >>= 8 * (q & 1);
  return w;
}

// The activation operand: 16 consecutive 16-bit values at p (zero when the
// lane's token does not exist).
__device__ __forceinline__ void load_b(const uint16_t* p, bool valid, uint32_t (&b)[8]) {
  uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
  if (valid) {
    v0 = *reinterpret_cast<const uint4*>(p);
    v1 = *reinterpret_cast<const uint4*>(p + 8);
  }
  b[0] = v0.x;
  b[1] = v0.y;
  b[2] = v0.z;
  b[3] = v0.w;
  b[4] = v1.x;
  b[5] = v1.y;
  b[6] = v1.z;
  b[7] = v1.w;
}

// Waits (bounded) until *slot, written by another warp of the CTA, reaches
// `job`; returns true when it gave up.
__device__ __forceinline__ bool issued2_wait(const int* slot, int job) {
  if (*reinterpret_cast<const volatile int*>(slot) >= job) return false;
  const long long t0 = clock64();
  while (*reinterpret_cast<const volatile int*>(slot) < job)
    if (clock64() - t0 > kWaitLimitCycles) return true;
  return false;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Every routing output, as the routing kernel writes it for one chunk: ids
// and weights, counts, exclusive offsets, the stable permutation and the tile
// block map (experts ascending).  Run by the compute warps of one CTA.
//   cnt: scratch of 3 * E + 2 ints in shared memory (E <= 256)
__device__ __forceinline__ void write_routing_outputs(const DecodeArgs& a, const int* s_ids, const float* s_w, int* cnt,
                                                   int na, int warp, int lane) {
  int* off = cnt + a.E;       // [E + 1]
  int* boff = off + a.E + 1;  // [E + 1]
  for (int i = threadIdx.x; i < na; i += kCons) {
    a.out.ids[i] = s_ids[i];
    a.out.w[i] = s_w[i];
  }
  for (int e = threadIdx.x; e < a.E; e += kCons) cnt[e] = 0;
  book_sync();
  for (int i = threadIdx.x; i < na; i += kCons) atomicAdd(&cnt[s_ids[i]], 1);
  book_sync();
  if (warp == 0) {
    int run = 0, brun = 0;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < a.E ? cnt[e] : 0;
      const int b = (c + a.block_rows - 1) / a.block_rows;
      int ic = c, ib = b;
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
  book_sync();
  for (int e = threadIdx.x; e < a.E; e += kCons) a.out.counts[e] = cnt[e];
  for (int e = threadIdx.x; e <= a.E; e += kCons) a.out.offsets[e] = off[e];
  for (int i = threadIdx.x; i < na; i += kCons) {
    const int e = s_ids[i];
    int r = 0;
    for (int j = 0; j < i; ++j) r += s_ids[j] == e;
    const int pos = off[e] + r;
    a.out.perm[pos] = i;
    a.out.inv_perm[i] = pos;
  }
  for (int e = threadIdx.x; e < a.E; e += kCons) {
    const int c = cnt[e];
    int b = boff[e];
    for (int r = 0; r < c; r += a.block_rows, ++b) {
      a.out.block_map[3 * b + 0] = e;
      a.out.block_map[3 * b + 1] = off[e] + r;
      a.out.block_map[3 * b + 2] = min(a.block_rows, c - r);
    }
  }
}

// Test hooks (moe_debug_decode): the limit of the wait at the barrier over the
// grid, in SM clock cycles, and one CTA whose arrival at that barrier is
// skipped, so that every CTA's wait runs out (a bounded wait that expires;
// nothing faults).
__device__ long long g_dec_wait_limit = kWaitLimitCycles;
__device__ int g_dec_drop_cta = -1;

// kReg: every CTA has at most one phase-1 item and d <= 64 * 8 * kRegChunks;
// the item's gate/up codes go from global memory straight into the MMA
// fragment registers of the warps that use them, loaded as soon as the
// item's expert is known (before the wait for the previous kernel for the
// shared expert), instead of through the phase-1 stage ring.
template <int kT, int kBits, bool kReg>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeMaps mr, const __grid_constant__ DecodeMaps ms, const DecodeArgs a,
                  WsHeader* hdr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int d = a.d;
  constexpr int kW = kWpg<kBits>;  // code words per row and group
  const Layout L = layout(kT, d, a.I, a.I_shared, kBits);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, q4 = lane & 3;  // MMA fragment row group and column pair
  const int nC = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const bool fused = a.logits != nullptr;
  const bool has_shared = a.I_shared > 0;
  const int rs0 = has_shared ? 1 : 0;
  const int it_r = a.I / kRows1, it_s = a.I_shared / kRows1;  // phase-1 items per routed / shared expert
  const int G2 = a.I / 64, G2s = a.I_shared / 64;               // phase-2 groups per routed / shared slot
  const int nrb = d / kRows2;
  const int my_rbs = cta < nrb ? div_up(nrb - cta, nC) : 0;
  const bool bookkeeper = fused && cta == nC - 1;

  uint8_t* ring1 = smem + L.ring1;
  uint8_t* ring2 = smem + L.ring2;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
  float* sx = reinterpret_cast<float*>(smem + L.sx);
  float* red1 = reinterpret_cast<float*>(smem + L.red1);
  float* red2 = reinterpret_cast<float*>(smem + L.red2);
  float* wt = reinterpret_cast<float*>(smem + L.wt);
  int* slot_e = reinterpret_cast<int*>(smem + L.slot_e);
  int* s_ids = reinterpret_cast<int*>(smem + L.rid);
  float* s_w = reinterpret_cast<float*>(smem + L.rid + static_cast<size_t>(kT) * kMaxK * 4);
  int* s_slot = reinterpret_cast<int*>(smem + L.rid + 2ull * kT * kMaxK * 4);
  int* misc = reinterpret_cast<int*>(smem + L.misc);
  int* cnt1 = reinterpret_cast<int*>(smem + L.cnt);
  int* cnt2 = cnt1 + kS1;
  int* issued2 = cnt2 + kS2Max;
  uint64_t* full1 = reinterpret_cast<uint64_t*>(smem + L.bars);  // phase-1 stage loaded
  uint64_t* empty1 = full1 + kS1;                                 // phase-1 stage consumed
  uint64_t* full2c = empty1 + kS1;                                // phase-2 stage: down rows loaded
  uint64_t* full2h = full2c + kS2Max;                             // phase-2 stage: h record loaded
  uint64_t* empty2 = full2h + kS2Max;                             // phase-2 stage consumed
  uint64_t* bar_x = empty2 + kS2Max;
  uint64_t* bar_w = bar_x + 1;   // the routing weights are in wt
  uint64_t* bar_h0 = bar_w + 1;  // the h records of the first min(S2, jobs) phase-2 jobs have landed
  uint8_t* hring = smem + L.hring;
  float* s_v = reinterpret_cast<float*>(smem + L.rid + 3ull * kT * kMaxK * 4);
  double* s_ex = reinterpret_cast<double*>(smem + round_up(L.rid + 4ull * kT * kMaxK * 4, 8));

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBars; ++i) mbar_init(&full1[i], 1);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < kS1 + kS2Max; i += kThreads) cnt1[i] = 0;
  for (int i = threadIdx.x; i < kS2Max; i += kThreads) issued2[i] = i;  // stage s first holds job s
  for (int i = threadIdx.x; i < kMaxSlots * kT; i += kThreads) wt[i] = 0.0f;
  __syncthreads();

  // ------------------------------------------------------------ loads (the producer warp)
  // Phase-1 job j of this CTA: chunk j % nchunk of its item j / nchunk.
  auto item_slot = [&](int it, int& slot, int& rb) {
    if (it < it_s) {
      slot = 0;
      rb = it;
    } else {
      const int v = it - it_s;
      slot = rs0 + v / it_r;
      rb = v % it_r;
    }
  };
  // The item's group parameters (every group of its 32 rows, both matrices)
  // come with its first chunk, into the parameter buffer of that chunk's
  // stage; the stage's next first chunk is issued only once this item has
  // been consumed, so the buffer lives as long as the item.
  auto issue1 = [&](int j) {
    const int stage = j % kS1, ch = j % L.nchunk, il = j / L.nchunk;
    int slot, rb;
    item_slot(cta + il * nC, slot, rb);
    const bool sh = has_shared && slot == 0;
    const int e = sh ? 0 : slot_e[slot];
    const DecodeMaps& m = sh ? ms : mr;
    uint8_t* st = ring1 + static_cast<size_t>(stage) * kSt1<kBits>;
    uint64_t* bar = &full1[stage];
    const uint32_t sbb = static_cast<uint32_t>(L.G1) * kRows1 * 4;
    mbar_arrive_expect_tx(bar, kSt1<kBits> + (ch == 0 ? 2 * sbb : 0u));
    tma_load_3d(st, &m.q_gate, bar, rb * kRows1 * kW, ch * kChunk, e);
    tma_load_3d(st + kCodeQ<kBits>, &m.q_up, bar, rb * kRows1 * kW, ch * kChunk, e);
    if (ch == 0) {
      uint8_t* sbd = smem + L.sbuf1 + static_cast<size_t>(stage) * L.sb1;
      tma_load_3d(sbd, &m.sb_gate, bar, rb * kRows1, 0, e);
      tma_load_3d(sbd + sbb, &m.sb_up, bar, rb * kRows1, 0, e);
    }
  };
  // Phase-2 job j2: slot j2 % nsl of the CTA's row block j2 / nsl.
  auto issue2c = [&](int j2, int nsl) {
    const int stage = j2 % L.S2, slot = j2 % nsl;
    const int rb = cta + (j2 / nsl) * nC;
    const bool sh = has_shared && slot == 0;
    const int e = sh ? 0 : slot_e[slot];
    const uint32_t gx = static_cast<uint32_t>(sh ? G2s : G2);
    const DecodeMaps& m = sh ? ms : mr;
    uint8_t* st = ring2 + static_cast<size_t>(stage) * L.st2;
    uint64_t* bar = &full2c[stage];
    mbar_arrive_expect_tx(bar, gx * kRows2 * (4 * kW + 4));
    tma_load_3d(st, &m.q_down, bar, rb * kRows2 * kW, 0, e);
    tma_load_3d(st + L.st2_sb, &m.sb_down, bar, rb * kRows2, 0, e);
  };
  auto issue2h = [&](int j2, int nsl) {
    const int stage = j2 % L.S2, slot = j2 % nsl;
    uint64_t* bar = &full2h[stage];
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(L.hrec));
    bulk_g2s(hring + static_cast<size_t>(stage) * L.hrec, a.hbuf + static_cast<size_t>(slot) * L.hrec,
             static_cast<uint32_t>(L.hrec), bar);
  };
  // The same copies issued by the whole producer warp at once, one copy per
  // lane (a warp issues copies about three times faster than one lane issuing
  // them in turn): first every barrier's byte count, then the copies.
  //   phase-1 jobs [j0, j0 + n), n <= 8: lane 4i + c issues copy c of job j0 + i
  //   (gate codes, up codes, gate parameters, up parameters; the last two with
  //   an item's first chunk only)
  auto issue1_warp = [&](int j0, int n) {
    const uint32_t sbb = static_cast<uint32_t>(L.G1) * kRows1 * 4;
    if (lane < n) {
      const int j = j0 + lane;
      mbar_arrive_expect_tx(&full1[j % kS1], kSt1<kBits> + (j % L.nchunk == 0 ? 2 * sbb : 0u));
    }
    __syncwarp();
    const int i = lane >> 2, c = lane & 3;
    const int j = j0 + i, ch = j % L.nchunk, il = j / L.nchunk;
    if (i < n && (c < 2 || ch == 0)) {
      int slot, rb;
      item_slot(cta + il * nC, slot, rb);
      const bool sh = has_shared && slot == 0;
      const int e = sh ? 0 : slot_e[slot];
      const DecodeMaps& m = sh ? ms : mr;
      const int stage = j % kS1;
      uint64_t* bar = &full1[stage];
      if (c < 2) {
        tma_load_3d(ring1 + static_cast<size_t>(stage) * kSt1<kBits> + c * kCodeQ<kBits>,
                    c == 0 ? &m.q_gate : &m.q_up, bar, rb * kRows1 * kW, ch * kChunk, e);
      } else {
        tma_load_3d(smem + L.sbuf1 + static_cast<size_t>(stage) * L.sb1 + (c - 2) * sbb, c == 2 ? &m.sb_gate : &m.sb_up,
                    bar, rb * kRows1, 0, e);
      }
    }
  };
  //   phase-2 jobs [j0, j0 + n), n <= 16: lane 2i + c issues the codes (c = 0) or
  //   the parameters (c = 1) of job j0 + i
  auto issue2c_warp = [&](int j0, int n, int nsl) {
    if (lane < n) {
      const int j2 = j0 + lane, slot = j2 % nsl;
      const uint32_t gx = static_cast<uint32_t>(has_shared && slot == 0 ? G2s : G2);
      mbar_arrive_expect_tx(&full2c[j2 % L.S2], gx * kRows2 * (4 * kW + 4));
    }
    __syncwarp();
    const int i = lane >> 1, c = lane & 1;
    if (i < n) {
      const int j2 = j0 + i, stage = j2 % L.S2, slot = j2 % nsl;
      const int rb = cta + (j2 / nsl) * nC;
      const bool sh = has_shared && slot == 0;
      const int e = sh ? 0 : slot_e[slot];
      const DecodeMaps& m = sh ? ms : mr;
      uint8_t* st = ring2 + static_cast<size_t>(stage) * L.st2;
      if (c == 0) tma_load_3d(st, &m.q_down, &full2c[stage], rb * kRows2 * kW, 0, e);
      else tma_load_3d(st + L.st2_sb, &m.sb_down, &full2c[stage], rb * kRows2, 0, e);
    }
  };

  // Register path: the item's group parameters (both matrices) by TMA into
  // the first parameter buffer, on the first stage's barrier (one lane).
  auto issue_params = [&](int slot, int rb) {
    const bool sh = has_shared && slot == 0;
    const int e = sh ? 0 : slot_e[slot];
    const DecodeMaps& m = sh ? ms : mr;
    const uint32_t sbb = static_cast<uint32_t>(L.G1) * kRows1 * 4;
    mbar_arrive_expect_tx(&full1[0], 2 * sbb);
    tma_load_3d(smem + L.sbuf1, &m.sb_gate, &full1[0], rb * kRows1, 0, e);
    tma_load_3d(smem + L.sbuf1 + sbb, &m.sb_up, &full1[0], rb * kRows1, 0, e);
  };
  // Register path: compute warp (matrix p1_mat, group p1_gl of each chunk)
  // loads the code words its MMA fragments take, rows g8, g8 + 8, g8 + 16 and
  // g8 + 24 of the item's 32 (codes [E][d/64][N][wpg], N = I or I_shared).
  const int p1_mat = warp >> 3, p1_gl = warp & 7;
  uint2 cw[kRegChunks][4];
  auto load_item_codes = [&](int slot, int rb) {
    const bool sh = has_shared && slot == 0;
    const int e = sh ? 0 : slot_e[slot];
    const int N = sh ? a.I_shared : a.I;
    const uint32_t* base = p1_mat == 0 ? (sh ? a.qg_s : a.qg_r) : (sh ? a.qu_s : a.qu_r);
    base += static_cast<size_t>(e) * L.G1 * N * kW;
#pragma unroll
    for (int ch = 0; ch < kRegChunks; ++ch) {
      const int gi = ch * kChunk + p1_gl;
      if (ch < L.nchunk && gi < L.G1) {
        const uint32_t* row = base + (static_cast<size_t>(gi) * N + rb * kRows1 + g8) * kW;
#pragma unroll
        for (int r = 0; r < 4; ++r) cw[ch][r] = ldg_codes<kBits>(row + ((r >> 1) * 16 + (r & 1) * 8) * kW, q4);
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) cw[ch][r] = make_uint2(0u, 0u);
      }
    }
  };

  // The shared expert's loads need no routing and do not depend on the
  // previous kernels: issue them first (the CTA's items come in index order,
  // the shared expert's first).  Tensor maps, router logits and X are only
  // pulled towards the SM (an L2 prefetch of a line the previous kernel still
  // writes is harmless: L2 is where writes land).
  const int my_sh_items = cta < it_s ? div_up(it_s - cta, nC) : 0;
  const int pre1 = kReg ? 0 : min(kS1, my_sh_items * L.nchunk);
  const int pre2 = has_shared && my_rbs > 0 ? 1 : 0;
  if (warp == kProducer) {
    if (kReg) {
      if (my_sh_items > 0 && lane == 0) issue_params(0, cta);
    } else {
      issue1_warp(0, pre1);
    }
    if (pre2) issue2c_warp(0, 1, 1);
    if (lane == 1) {
      tma_prefetch_desc(&mr.q_gate);
      tma_prefetch_desc(&mr.q_up);
      tma_prefetch_desc(&mr.sb_gate);
      tma_prefetch_desc(&mr.sb_up);
      tma_prefetch_desc(&mr.q_down);
      tma_prefetch_desc(&mr.sb_down);
    } else if (lane == 2 && has_shared) {
      tma_prefetch_desc(&ms.q_gate);
      tma_prefetch_desc(&ms.q_up);
      tma_prefetch_desc(&ms.sb_gate);
      tma_prefetch_desc(&ms.sb_up);
      tma_prefetch_desc(&ms.q_down);
      tma_prefetch_desc(&ms.sb_down);
    }
  } else if (warp == 1) {
    // Loads (values unused) bring the router logits and X into L2 now; they
    // are read for use after the wait (L2 is where a write by the previous
    // kernel lands, so a line fetched early is never stale there).
    const char* lg = reinterpret_cast<const char*>(a.logits);
    const char* xp = reinterpret_cast<const char*>(a.X);
    if (lg)
      for (int off = lane * 128; off < kT * a.E * 4; off += 32 * 128) touch_l2(lg + off);
    for (int off = lane * 128; off < kT * d * 2; off += 32 * 128) touch_l2(xp + off);
  }
  if (kReg && warp < kWarps && my_sh_items > 0) load_item_codes(0, cta);  // a shared-expert item: rows 32 cta ..
  pdl_wait();  // X, the routing and the previous layer's use of the workspace
  // Call g of this workspace counts barrier arrivals in dec_count[g % 2]; read
  // before the CTA's first barrier so it precedes every arrival of the call.
  const uint32_t gen = *reinterpret_cast<volatile uint32_t*>(&hdr->dec_gen);

  if (threadIdx.x == 32 * kGemvMaxT) {  // X into shared memory
    mbar_arrive_expect_tx(bar_x, static_cast<uint32_t>(kT * d * 2));
    bulk_g2s(xs, a.X, static_cast<uint32_t>(kT * d * 2), bar_x);
  }

  // ------------------------------------------------------------ routing
  const int na = kT * a.k;
  bool ok = true;  // every wait completed
  float sel_v = 0.0f;  // fused routing: this lane's selected logit (warps < T)
  if (warp < kT) {
    if (fused) {
      int sel_i;
      bool finite;
      warp_topk_select<8>(a.logits + static_cast<size_t>(warp) * a.E, a.E, a.k, lane, sel_i, sel_v, finite);
      if (bookkeeper && !finite && lane == 0) record_status(a.status, MOE_ERR_NONFINITE);
      if (lane < a.k) {
        s_ids[warp * a.k + lane] = sel_i;
        s_v[warp * a.k + lane] = sel_v;
      }
    } else {
      for (int i = lane; i < a.k; i += 32) {
        s_ids[warp * a.k + i] = __ldcg(a.ids + warp * a.k + i);
        s_w[warp * a.k + i] = __ldcg(a.w + warp * a.k + i);
      }
    }
    if (kT > 1) asm volatile("bar.sync 3, %0;" ::"r"(32 * kT) : "memory");
    if (warp == 0) {
      // Distinct experts of the call in order of first appearance.
      __syncwarp();
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
      if (has_shared && lane == 0) slot_e[0] = 0;
      if (lane == 0) misc[0] = nsl - rs0;
      __syncwarp();
      if (!fused) {  // weights read from memory are placed now
        for (int i = lane; i < na; i += 32) wt[s_slot[i] * kT + i / a.k] = s_w[i];
        if (has_shared && lane < kT) wt[lane] = 1.0f;
      }
    }
  }
  __syncthreads();  // the slots are known
  const int nsl_r = misc[0];
  const int nsl = rs0 + nsl_r;
  pdl_launch_dependents();
  const int NI = it_s + nsl_r * it_r;
  const int my_items = cta < NI ? div_up(NI - cta, nC) : 0;
  const int total1 = my_items * L.nchunk;
  const int total2 = my_rbs * nsl;
  if (kReg) {
    if (NI > nC && cta == 0 && threadIdx.x == 0) record_status(a.status, MOE_ERR_UNSUPPORTED);  // never: the host checks
    if (warp < kWarps && my_sh_items == 0 && my_items > 0) {  // a routed item
      int slot, rb;
      item_slot(cta, slot, rb);
      load_item_codes(slot, rb);
    }
  }

  if (warp == kProducer) {
    // -------------------------------------------------------- producer
    // Every copy of the CTA, in the order the compute warps use them: the
    // gate/up chunks (refilling a stage once the compute warps have released
    // it), the down rows, then, after the barrier over the grid, the h
    // records.  Issuing a copy waits while the SM's copy queue is full, so no
    // compute warp issues any.
    if (kReg) {
      if (my_sh_items == 0 && my_items > 0 && lane == 0) {
        int slot, rb;
        item_slot(cta, slot, rb);
        issue_params(slot, rb);
      }
      // The down rows too, at once: the gate/up codes do not wait for the
      // copy queue here, and the down rows then land during phase 1 (measured:
      // 40-layer step 0.466 -> 0.454 ms against issuing them after phase 1).
      __syncwarp();
      for (int j0 = pre2, n2 = min(L.S2, total2); j0 < n2; j0 += 16) issue2c_warp(j0, min(16, n2 - j0), nsl);
    } else {
      issue1_warp(pre1, min(kS1, total1) - pre1);
    }
    // The routing weights (fp64, slow on this GPU), while the copies stream:
    // softmax over each token's selected logits, summed in selection order and
    // rounded once (the routing kernel's arithmetic, so the same bits).
    if (fused) {
      for (int i = lane; i < na; i += 32)
        s_ex[i] = exp(static_cast<double>(s_v[i]) - static_cast<double>(s_v[(i / a.k) * a.k]));
      __syncwarp();
      for (int i = lane; i < na; i += 32) {
        double sum = 0.0;
        for (int j = 0; j < a.k; ++j) sum += s_ex[(i / a.k) * a.k + j];
        wt[s_slot[i] * kT + i / a.k] = static_cast<float>(s_ex[i] / sum);
      }
      if (has_shared && lane < kT) wt[lane] = 1.0f;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_w);  // releases the weights to the compute warps
    if (!kReg && lane == 0) {
      for (int j = kS1; j < total1; ++j) {
        ok &= mbar_wait(&empty1[j % kS1], static_cast<uint32_t>(j / kS1 - 1) & 1u, nullptr);
        issue1(j);
      }
    }
    // Ring path: the down rows, once this CTA's last gate/up chunk has landed:
    // the gate/up bytes, on the path to the barrier over the grid, take the
    // memory bandwidth first; the down rows are needed only after that barrier.
    __syncwarp();
    if (!kReg) {
      if (total1 > 0)
        ok &= mbar_wait(&full1[(total1 - 1) % kS1], static_cast<uint32_t>((total1 - 1) / kS1) & 1u, nullptr);
      for (int j0 = pre2, n2 = min(L.S2, total2); j0 < n2; j0 += 16) issue2c_warp(j0, min(16, n2 - j0), nsl);
    }
    if (lane == 0) {
      // the barrier: every CTA has written its h records.  CTA 0 then clears
      // the other counter (last used by call g - 1, which has finished) and
      // advances the call number for call g + 1 (read only after this call).
      uint32_t* count = &hdr->dec_count[gen & 1u];
      const long long t0 = clock64();
      while (ld_acquire_gpu(count) < static_cast<uint32_t>(nC)) {
        if (clock64() - t0 > g_dec_wait_limit) {
          record_status(a.status, MOE_ERR_TIMEOUT);
          break;
        }
      }
      if (cta == 0) {
        hdr->dec_count[(gen + 1) & 1u] = 0;
        hdr->dec_gen = gen + 1;
      }
    }
    if (lane == 0) {
      // the h records of jobs [0, n0): consecutive jobs of one row block are
      // consecutive slots, so each run is one copy into consecutive stages
      fence_proxy_async_global();
      const int n0 = min(L.S2, total2);
      if (n0 > 0) {
        mbar_arrive_expect_tx(bar_h0, static_cast<uint32_t>(n0 * L.hrec));
        for (int j = 0; j < n0;) {
          const int run = min(nsl - j % nsl, n0 - j);
          bulk_g2s(hring + static_cast<size_t>(j) * L.hrec, a.hbuf + static_cast<size_t>(j % nsl) * L.hrec,
                   static_cast<uint32_t>(run * L.hrec), bar_h0);
          j += run;
        }
      }
      for (int j2 = L.S2; j2 < total2; ++j2) {
        const int stage = j2 % L.S2;
        ok &= mbar_wait(&empty2[stage], static_cast<uint32_t>(j2 / L.S2 - 1) & 1u, nullptr);
        *reinterpret_cast<volatile int*>(issued2 + stage) = j2;
        issue2c(j2, nsl);
        issue2h(j2, nsl);
      }
    }
  } else {
    // -------------------------------------------------------- compute warps
    {
      // sums of x over each group of 64 columns, 8 threads per (token, group)
      const int t0 = threadIdx.x - 32 * (kGemvMaxT + 1);
      if (t0 >= 0) {
        ok &= mbar_wait(bar_x, 0, nullptr);
        constexpr int kSum = kCons - 32 * (kGemvMaxT + 1);
        for (int i = t0; i < div_up(kT * L.G1 * 8, kSum) * kSum; i += kSum) {
          const int pair = i >> 3, part = i & 7;
          float v = 0.0f;
          if (pair < kT * L.G1) {
            const int t = pair / L.G1, gi = pair % L.G1;
            const uint4 u = *reinterpret_cast<const uint4*>(xs + static_cast<size_t>(t) * d + gi * 64 + part * 8);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) v += bf16_lo(w[c]) + bf16_hi(w[c]);
          }
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          if (pair < kT * L.G1 && part == 0) sx[pair] = v;
        }
      }
    }
    cons_sync();

    // ------------------------------------------------------------ phase 1: h of this CTA's items
    const int mat = warp >> 3;  // 0: gate, 1: up
    const int gl = warp & 7;    // group inside a stage
    const int n_items = kReg ? min(my_items, 1) : my_items;
    for (int il = 0; il < n_items; ++il) {
      int slot, rb;
      item_slot(cta + il * nC, slot, rb);
      const uint32_t* sbi =
          reinterpret_cast<const uint32_t*>(smem + L.sbuf1 + static_cast<size_t>((il * L.nchunk) % kS1) * L.sb1) +
          mat * L.G1 * kRows1;
      float acc[2][4];  // [tile][fragment]
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[0][i] = acc[1][i] = 0.0f;
      // group gi of the item: the MMAs of both 16-row tiles (codes of rows
      // g8, g8 + 8, g8 + 16, g8 + 24 in w4), then the group's affine map
      auto group1 = [&](int gi, const uint2 (&w4)[4]) {
        const uint32_t* sbm = sbi + gi * kRows1;
        uint32_t b[8];
        load_b(xs + static_cast<size_t>(g8) * d + gi * 64 + 16 * q4, g8 < kT, b);
        const float sxa = 2 * q4 < kT ? sx[(2 * q4) * L.G1 + gi] : 0.0f;
        const float sxb = 2 * q4 + 1 < kT ? sx[(2 * q4 + 1) * L.G1 + gi] : 0.0f;
        float dd[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) mma_group<true, kBits>(w4[2 * tile], w4[2 * tile + 1], b, dd[tile]);
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
          const int r0 = tile * 16 + g8;
          const uint32_t p0 = sbm[r0], p1 = sbm[r0 + 8];
          const float s0 = bf16_lo(p0), c0 = bf16_hi(p0) - 128.0f * s0;
          const float s1 = bf16_lo(p1), c1 = bf16_hi(p1) - 128.0f * s1;
          acc[tile][0] += fmaf(s0, dd[tile][0], c0 * sxa);
          acc[tile][1] += fmaf(s0, dd[tile][1], c0 * sxb);
          acc[tile][2] += fmaf(s1, dd[tile][2], c1 * sxa);
          acc[tile][3] += fmaf(s1, dd[tile][3], c1 * sxb);
        }
      };
      if constexpr (kReg) {
        ok &= mbar_wait(&full1[0], 0, nullptr);  // the item's group parameters
#pragma unroll
        for (int ch = 0; ch < kRegChunks; ++ch) {
          const int gi = ch * kChunk + gl;
          if (ch < L.nchunk && gi < L.G1) {
            uint2 w4[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) w4[r] = codes_fix<kBits>(cw[ch][r], q4);
            group1(gi, w4);
          }
        }
      } else {
        for (int ch = 0; ch < L.nchunk; ++ch) {
          const int j = il * L.nchunk + ch, stage = j % kS1;
          ok &= mbar_wait(&full1[stage], static_cast<uint32_t>(j / kS1) & 1u, nullptr);
          const int gi = ch * kChunk + gl;  // this warp's group
          if (gi < L.G1) {
            const uint32_t* qm = reinterpret_cast<const uint32_t*>(ring1 + static_cast<size_t>(stage) * kSt1<kBits> +
                                                                   mat * kCodeQ<kBits>) +
                                 gl * kRows1 * kW;
            uint2 w4[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) w4[r] = load_codes<kBits>(qm + ((r >> 1) * 16 + (r & 1) * 8 + g8) * kW, q4);
            group1(gi, w4);
          }
          // the last warp done with a stage releases it to the producer
          __syncwarp();
          if (lane == 0 && (atomicAdd(&cnt1[stage], 1) + 1) % kWarps == 0) mbar_arrive(&empty1[stage]);
        }
      }
      // h of the item's 32 features for every token
#pragma unroll
      for (int tile = 0; tile < 2; ++tile) {
        float* rp = red1 + (warp * kRows1 + tile * 16 + g8) * kT;
        if (2 * q4 < kT) {
          rp[2 * q4] = acc[tile][0];
          rp[8 * kT + 2 * q4] = acc[tile][2];
        }
        if (2 * q4 + 1 < kT) {
          rp[2 * q4 + 1] = acc[tile][1];
          rp[8 * kT + 2 * q4 + 1] = acc[tile][3];
        }
      }
      cons_sync();
      if (warp < kT) {
        const int t = warp, r = lane;
        float gs = 0.0f, us = 0.0f;
#pragma unroll
        for (int w = 0; w < kChunk; ++w) {
          gs += red1[(w * kRows1 + r) * kT + t];
          us += red1[((kChunk + w) * kRows1 + r) * kT + t];
        }
        const __half hh = __float2half_rn(gs / (1.0f + expf(-gs)) * us);
        uint8_t* rec = a.hbuf + static_cast<size_t>(slot) * L.hrec;
        reinterpret_cast<__half*>(rec)[t * L.Imax + rb * kRows1 + r] = hh;
        float hsum = __half2float(hh);  // the sum of the values the MMA sees
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) hsum += __shfl_xor_sync(0xffffffffu, hsum, o);
        if (lane == 0)
          reinterpret_cast<float*>(rec + static_cast<size_t>(kT) * L.Imax * 2)[t * L.hs_stride + rb] = hsum;
      }
      cons_sync();
    }

    // ------------------------------------------------------------ arrival at the barrier over the grid
    // Every CTA of the launch is resident (one per SM, the grid is capped at
    // what fits); the h records written with ordinary stores are read by bulk
    // copies after it.
    fence_proxy_async_global();
    cons_sync();
    if (threadIdx.x == 0 && cta != g_dec_drop_cta) red_release_gpu_add(&hdr->dec_count[gen & 1u], 1u);

    // One CTA writes every routing output, after it has arrived (no CTA of the
    // call reads them): its own copy of the weights, from the same arithmetic
    // as the producer's.
    if (bookkeeper) {
      if (warp < kT) {
        const float w = warp_topk_weights(sel_v, a.k, lane);
        if (lane < a.k) s_w[warp * a.k + lane] = w;
      }
      book_sync();  // the weights are in s_w
      write_routing_outputs(a, s_ids, s_w, reinterpret_cast<int*>(smem + L.bk), na, warp, lane);
    }

    // ------------------------------------------------------------ phase 2: Y rows of this CTA
    // Warp w takes a contiguous run of the (slot, group) pairs of each row
    // block: it waits for and releases each slot's stage once.
    const int G2first = has_shared ? G2s : G2;  // groups of slot 0
    const int pairs = (has_shared ? G2s : 0) + nsl_r * G2;
    const int p_begin = warp * pairs / kWarps, p_end = (warp + 1) * pairs / kWarps;
    int s_begin = 0, g_begin = p_begin;
    if (p_begin >= G2first) {
      s_begin = 1 + (p_begin - G2first) / G2;
      g_begin = (p_begin - G2first) % G2;
    }
    // lane-constant offsets: codes of rows g8 and g8 + 8 (words), h of token g8 (halves)
    const int lq = g8 * kW;
    const size_t lh = static_cast<size_t>(g8) * L.Imax + 16 * q4;
    const bool refills = total2 > L.S2;
    for (int rl = 0; rl < my_rbs; ++rl) {
      const int rb = cta + rl * nC;
      float acc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      int slot = s_begin, gr = g_begin;
      int stage = (rl * nsl + s_begin) % L.S2, use = (rl * nsl + s_begin) / L.S2;  // job rl * nsl + slot
      for (int p = p_begin; p < p_end; ++slot, gr = 0) {
        const int j2 = rl * nsl + slot;
        const int gx = slot == 0 ? G2first : G2;
        const int g_stop = min(gx, gr + (p_end - p));
        // A warp may reach a job two uses of its stage ahead of the job the
        // stage holds, where the parity wait would pass on the older phase:
        // with refills, first wait until the job has been issued.
        if (refills && issued2_wait(issued2 + stage, j2)) ok = false;
        ok &= mbar_wait(&full2c[stage], static_cast<uint32_t>(use) & 1u, nullptr);
        if (j2 < L.S2) ok &= mbar_wait(bar_h0, 0, nullptr);
        else ok &= mbar_wait(&full2h[stage], static_cast<uint32_t>(use - 1) & 1u, nullptr);
        const uint8_t* st = ring2 + static_cast<size_t>(stage) * L.st2;
        const uint8_t* hr = hring + static_cast<size_t>(stage) * L.hrec;
        const uint32_t* qm = reinterpret_cast<const uint32_t*>(st) + lq;
        const uint32_t* sbm = reinterpret_cast<const uint32_t*>(st + L.st2_sb) + g8;
        const uint16_t* hp = reinterpret_cast<const uint16_t*>(hr) + lh;
        const float* hsa = reinterpret_cast<const float*>(hr + static_cast<size_t>(kT) * L.Imax * 2) + (2 * q4) * L.hs_stride;
        const float* hsb = hsa + L.hs_stride;
        float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // the slot's rows before its routing weight
        // one group of 64 columns: four MMA steps, then the group's affine map
        auto group = [&](int g, float (&dd)[4]) {
          uint32_t b[8];
          load_b(hp + g * 64, g8 < kT, b);
          const uint2 wa = load_codes<kBits>(qm + g * kRows2 * kW, q4);
          const uint2 wb = load_codes<kBits>(qm + g * kRows2 * kW + 8 * kW, q4);
          mma_group<false, kBits>(wa, wb, b, dd);
        };
        auto fold = [&](int g, const float (&dd)[4]) {
          const uint32_t p0 = sbm[g * kRows2], p1 = sbm[g * kRows2 + 8];
          const float s0 = bf16_lo(p0), c0 = bf16_hi(p0) - 1024.0f * s0;
          const float s1 = bf16_lo(p1), c1 = bf16_hi(p1) - 1024.0f * s1;
          const float ha = 2 * q4 < kT ? hsa[2 * g] + hsa[2 * g + 1] : 0.0f;
          sa[0] += fmaf(s0, dd[0], c0 * ha);
          sa[2] += fmaf(s1, dd[2], c1 * ha);
          if (kT > 1) {
            const float hb = 2 * q4 + 1 < kT ? hsb[2 * g] + hsb[2 * g + 1] : 0.0f;
            sa[1] += fmaf(s0, dd[1], c0 * hb);
            sa[3] += fmaf(s1, dd[3], c1 * hb);
          }
        };
        int g = gr;
        for (; g + 1 < g_stop; g += 2) {  // two groups in flight
          float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          group(g, d0);
          group(g + 1, d1);
          fold(g, d0);
          fold(g + 1, d1);
        }
        if (g < g_stop) {
          float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          group(g, d0);
          fold(g, d0);
        }
        // tokens not routed to the slot contribute nothing (their h is never used)
        if (slot == s_begin) ok &= mbar_wait(bar_w, 0, nullptr);
        const float ra = 2 * q4 < kT ? wt[slot * kT + 2 * q4] : 0.0f;
        if (ra != 0.0f) {
          acc2[0] = fmaf(ra, sa[0], acc2[0]);
          acc2[2] = fmaf(ra, sa[2], acc2[2]);
        }
        if (kT > 1) {
          const float rb2 = 2 * q4 + 1 < kT ? wt[slot * kT + 2 * q4 + 1] : 0.0f;
          if (rb2 != 0.0f) {
            acc2[1] = fmaf(rb2, sa[1], acc2[1]);
            acc2[3] = fmaf(rb2, sa[3], acc2[3]);
          }
        }
        // the last warp done with a stage releases it to the producer (only
        // needed when some job waits for a stage)
        const int done = g_stop - gr;
        p += done;
        if (refills) {
          __syncwarp();
          if (lane == 0) {
            const int old = atomicAdd(&cnt2[stage], done);
            int need = 0;  // pairs of every job this stage has held, up to this one
            for (int jj = stage; jj <= j2; jj += L.S2) need += jj % nsl == 0 ? G2first : G2;
            if (old + done == need) mbar_arrive(&empty2[stage]);
          }
        }
        if (++stage == L.S2) {
          stage = 0;
          ++use;
        }
      }
      if (2 * q4 < kT) {
        red2[(warp * kRows2 + g8) * kT + 2 * q4] = acc2[0];
        red2[(warp * kRows2 + g8 + 8) * kT + 2 * q4] = acc2[2];
      }
      if (2 * q4 + 1 < kT) {
        red2[(warp * kRows2 + g8) * kT + 2 * q4 + 1] = acc2[1];
        red2[(warp * kRows2 + g8 + 8) * kT + 2 * q4 + 1] = acc2[3];
      }
      cons_sync();
      // Y = the sum over the 16 warps' partial rows: 8 lanes per output value
      // add pairs of partials, then a fixed shuffle tree (deterministic)
      if (threadIdx.x < kRows2 * kT * 8) {
        const int w8 = threadIdx.x & 7, o = threadIdx.x >> 3;  // output o = r * kT + t
        float v = red2[w8 * kRows2 * kT + o] + red2[(w8 + 8) * kRows2 * kT + o];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        if (w8 == 0) {
          const int r = o / kT, t = o % kT;
          a.Y[static_cast<size_t>(t) * d + rb * kRows2 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
      }
      cons_sync();
    }
  }
  if (!ok) record_status(a.status, MOE_ERR_TIMEOUT);
}

// CTAs of this kernel that can be resident at once on the current device (0
// on error).  The barrier over the grid needs every CTA resident together.
template <int kT, int kBits, bool kReg>
int max_ctas(size_t smem, int num_sms) {
  const void* f = reinterpret_cast<const void*>(decode_kernel<kT, kBits, kReg>);
  if (set_max_dynamic_smem(f, static_cast<int>(kSmemMax)) != cudaSuccess) return 0;
  int per_sm = 0;
  if (occupancy_per_sm(f, kThreads, smem, &per_sm) != cudaSuccess) return 0;
  return per_sm * num_sms;
}

template <int kT, int kBits, bool kReg>
cudaError_t launch_k(const DecodeArgs& a, const DecodeMaps* routed, const DecodeMaps* sh, WsHeader* hdr, int grid,
                     size_t smem, cudaStream_t stream, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  return cudaLaunchKernelEx(&cfg, decode_kernel<kT, kBits, kReg>, *routed, *sh, a, hdr);
}

// items: phase-1 items of the call at most.  One token whose items fit the
// grid (one per CTA) and d <= 2048 takes the register-load variant unless
// MOE_DECODE_REG=0.
template <int kT, int kBits>
cudaError_t launch_t(const DecodeArgs& a, const DecodeMaps* routed, const DecodeMaps* sh, WsHeader* hdr, int want,
                     size_t smem, cudaStream_t stream, bool pdl, int items) {
  if constexpr (kT == 1) {
    const char* env = std::getenv("MOE_DECODE_REG");
    const bool allow = !(env && env[0] == '0');
    if (allow && a.d <= 64 * kDecodeChunkGroups * kRegChunks) {
      const int resident = max_ctas<1, kBits, true>(smem, a.num_sms);
      if (resident < 1) return cudaErrorInvalidConfiguration;
      const int grid = want < resident ? want : resident;
      if (items <= grid) return launch_k<1, kBits, true>(a, routed, sh, hdr, grid, smem, stream, pdl);
    }
  }
  const int resident = max_ctas<kT, kBits, false>(smem, a.num_sms);
  if (resident < 1) return cudaErrorInvalidConfiguration;
  const int grid = want < resident ? want : resident;
  return launch_k<kT, kBits, false>(a, routed, sh, hdr, grid, smem, stream, pdl);
}

}  // namespace

bool decode_supported(int T, int d, int I, int I_shared, int k) {
  if (T < 1 || T > kGemvMaxT || k > kMaxK || k < 1) return false;
  if (d % 64 || I % 64 || I_shared % 64 || I < 64) return false;
  const int Imax = I > I_shared ? I : I_shared;
  if (Imax / 64 > 256 || d / 64 > 256) return false;  // a parameter box covers every group of a row block
  const Layout L = layout(T, d, I, I_shared, 4);  // 2-bit codes need less shared memory
  return L.S2 >= 2 && L.total <= kSmemMax;
}

size_t decode_scratch_bytes(int T, int I, int I_shared) {
  const int Imax = I > I_shared ? I : I_shared;
  const size_t hs = round_up(Imax / 32, 4);
  return static_cast<size_t>(kMaxSlots) * (static_cast<size_t>(T) * Imax * 2 + static_cast<size_t>(T) * hs * 4);
}

template <int kBits>
cudaError_t launch_bits(const DecodeArgs& a, const DecodeMaps* routed, const DecodeMaps* sh, WsHeader* hdr, int want,
                        size_t smem, cudaStream_t stream, bool pdl, int items) {
  switch (a.T) {
    case 1: return launch_t<1, kBits>(a, routed, sh, hdr, want, smem, stream, pdl, items);
    case 2: return launch_t<2, kBits>(a, routed, sh, hdr, want, smem, stream, pdl, items);
    case 3: return launch_t<3, kBits>(a, routed, sh, hdr, want, smem, stream, pdl, items);
    default: return launch_t<4, kBits>(a, routed, sh, hdr, want, smem, stream, pdl, items);
  }
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodeMaps* routed, const DecodeMaps* shared, void* ws,
                          cudaStream_t stream, bool pdl) {
  if (!decode_supported(a.T, a.d, a.I, a.I_shared, a.k)) return cudaErrorInvalidValue;
  if (reinterpret_cast<uintptr_t>(a.hbuf) & 15u) return cudaErrorInvalidValue;
  if (a.bits < 2 || a.bits > 4) return cudaErrorInvalidValue;
  const Layout L = layout(a.T, a.d, a.I, a.I_shared, a.bits);
  const DecodeMaps* sh = shared ? shared : routed;  // never read without a shared expert
  const int distinct = a.T * a.k < a.E ? a.T * a.k : a.E;
  const int items = a.I_shared / kRows1 + distinct * (a.I / kRows1);
  const int rbs = a.d / kRows2;
  int want = items > rbs ? items : rbs;
  if (a.logits) want += 1;  // a CTA with no item writes the routing outputs when the grid has room
  if (want > a.num_sms) want = a.num_sms;
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  timer_begin(kKDecode, stream);
  cudaError_t err;
  if (a.bits == 2)
    err = launch_bits<2>(a, routed, sh, hdr, want, L.total, stream, pdl, items);
  else if (a.bits == 3)
    err = launch_bits<3>(a, routed, sh, hdr, want, L.total, stream, pdl, items);
  else
    err = launch_bits<4>(a, routed, sh, hdr, want, L.total, stream, pdl, items);
  timer_end(kKDecode, stream);
  return err;
}

cudaError_t decode_debug(long long wait_limit_cycles, int drop_cta) {
  const long long lim = wait_limit_cycles > 0 ? wait_limit_cycles : kWaitLimitCycles;
  cudaError_t e = cudaMemcpyToSymbol(g_dec_wait_limit, &lim, sizeof(lim));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_dec_drop_cta, &drop_cta, sizeof(drop_cta));
}

}  // namespace bm
