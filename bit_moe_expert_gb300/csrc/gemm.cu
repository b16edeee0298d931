// Prefill path: grouped expert GEMMs on the 5th-generation tensor cores with
// the 4-bit dequantisation fused in ("Perplexity's Lily Beats MLX-LM on
// MacBook M5", section "Prefill: keep routing on the GPU, dequantize in
// flight": the grouped GEMM dequantises one small tile at a time on chip,
// accumulates in FP32, writes bf16 and never materialises the expanded
// weights; the expert input projections are fused with the gate activation and
// the output projection with the routing scores and the shared expert).  Here
// SwiGLU is fused into the gate/up epilogue; the routing scores and the shared
// expert are applied by a separate combine kernel after the down GEMM (a
// combine fused into the down epilogue serialised on the shared expert's
// items, which every token waits for, and ran 2.3x slower).
//
// Operands are fp16 (the pages' Metal kernels use bf16): fp16 holds the
// dequantised weights of this format exactly and rounds h and X 8x more finely,
// at the same tensor-core rate; X is converted as it is gathered into the
// routing's row order.
//
// sm_103a design ("swap AB"): the weights are the M = 128 operand and an
// expert's tokens the N operand (16..128, a multiple of 16), so an expert with
// few tokens still streams its weight tile exactly once.  The dequantised
// weight tile never touches shared memory: dequantisation warps turn the TMA-
// loaded codes into fp16 and store them with tcgen05.st straight into tensor
// memory, where tcgen05.mma reads them as its A operand; shared memory carries
// only the packed codes, the group parameters and the token tile (TMA boxes of
// the gathered fp16 X, or of h).  Accumulators live in tensor memory.  A
// pipeline stage covers two quantisation groups (K = 128).
//
// Roles (one persistent CTA per SM):
//   warp 0       TMA producer (token tile, codes, group parameters)
//   warps 1-2    MMA issuers (gate and up matrices; the down GEMM uses one),
//                one elected lane each
//   warps 3-     epilogue (gate/up: 12 warps, down: 8): TMEM -> registers ->
//                SwiGLU and fp16 h (gate/up) or the fp32 expert-output rows,
//                staged in shared memory and stored by TMA (down)
//   then         dequantise codes -> fp16 A tiles in TMEM: four warps per
//                matrix (gate/up: 8, down: 4), one per quarter of the rows
// Synchronisation is by mbarriers; every wait is bounded (2 s) and records
// MOE_ERR_TIMEOUT instead of hanging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bm {

namespace {

// Warp roles.
constexpr int kProducerWarp = 0;   // TMA of codes and group parameters; cp.async gather of the token tile
constexpr int kMmaWarp0 = 1;       // two MMA issuers (warps 1 and 2)
constexpr int kEpiWarp0 = 3;       // epilogue warps from 3 (Cfg::kEpiWarps of them), then the dequantisation warps
constexpr uint32_t kBarEpilogue = 1;  // named barrier of the epilogue warps (0 is __syncthreads)
constexpr uint32_t kTmemCols = 512;
static_assert(kGemmBN % 16 == 0, "epilogue warps drain columns 16 at a time");

template <bool kGateUp, int kBits>
struct Cfg {
  static constexpr int kMats = kGateUp ? 2 : 1;
  static constexpr int kG = kGateUp ? kGemmGroupsGU : kGemmGroupsDown;  // quantisation groups (K = 64) per stage
  // epilogue warps: two or three per TMEM lane quarter, each draining kEpiCols columns of the tile.  The
  // gate/up GEMM's single accumulator holds the next item's products back during its epilogue, so it takes
  // three (49.9 against 51.7 us for the long-prefill chunk); the down GEMM's epilogue overlaps them.
  static constexpr int kEpiWarps = kGateUp ? 12 : 8;
  static constexpr int kEpiCols = 16 * ((kGemmBN / 16 + kEpiWarps / 4 - 1) / (kEpiWarps / 4));
  static constexpr int kDqWarp0 = kEpiWarp0 + kEpiWarps;  // four dequantisation warps per matrix, one per lane quarter
  static constexpr int kDqWarps = 4 * kMats;
  static constexpr int kThreads = (kDqWarp0 + kDqWarps) * 32;
  static constexpr int kStages = 4;
  static constexpr int kAStages = kGateUp ? 2 : 4;
  static constexpr int kACols = 32 * kMats * kG;  // 64 fp16 per lane per matrix and group = 32 columns
  // accumulators: gate|up in one buffer (the gate/up GEMM's two-group A stages
  // leave TMEM room for one), the down GEMM's in two, so that its epilogue
  // overlaps the next item's products
  static constexpr int kAccBufs = kGateUp ? 1 : 2;
  static constexpr int kAccBufCols = kMats * kGemmBN;
  static constexpr int kABase = kAccBufs * kAccBufCols;
  static_assert(kABase + kAStages * kACols <= static_cast<int>(kTmemCols), "TMEM budget");
  static constexpr int kMmaIssuers = kMats;  // gate/up: one per matrix; down: one
  // token tile: one box of up to kGemmBN rows x 64 fp16 (128-byte swizzle) per group
  static constexpr int kBBoxBytes = kGemmBN * 128;
  static constexpr int kBBytes = kBBoxBytes * kG;
  // per group, 128 rows x (2 kBits) code words: 4-bit codes with a 32-byte swizzle, 2- and 3-bit codes (16
  // or 24 bytes a row) plain
  static constexpr int kQBytesG = kGemmBM * 8 * kBits;
  static constexpr int kQBytes = kQBytesG * kG;
  static constexpr int kSBBytesG = kGemmBM * 4;
  static constexpr int kSBBytes = kSBBytesG * kG;
  static constexpr int kStageTxBytes = kBBytes + kMats * (kQBytes + kSBBytes);
  static constexpr int kStageBytes = (kStageTxBytes + 1023) / 1024 * 1024;
  // down GEMM epilogue: per epilogue warp two staging buffers of [16 tokens][32 rows] fp32 for its TMA stores
  static constexpr int kEpiBufFloats = 16 * 32;
  static constexpr int kEpiStageBytes = kGateUp ? 0 : kEpiWarps * 2 * kEpiBufFloats * 4;
  static constexpr int kSmemBytes = kStages * kStageBytes + kEpiStageBytes + 1024 /*barriers etc.*/ + 1024 /*align*/;
  static constexpr int kEmptyArrivals = kDqWarps + kMmaIssuers;  // dequant warps + MMA commits
  static constexpr int kAEmptyArrivals = kMmaIssuers;
};

struct Item {
  int e, row0, rows, mt, nk;  // nk: quantisation groups along K
  bool shared;
  bool ok;  // false: a malformed block-map entry; every role skips it
};

struct Sched {
  int nb, mt_r, mt_s, n_routed, n_total, nsb;
};

__device__ __forceinline__ Item get_item(const GemmArgs& a, const Sched& s, int it, bool gate_up) {
  Item m;
  if (it < s.n_routed) {
    const int blk = it / s.mt_r;
    m.mt = it % s.mt_r;
    m.e = __ldg(a.block_map + 3 * blk + 0);
    m.row0 = __ldg(a.block_map + 3 * blk + 1);
    m.rows = __ldg(a.block_map + 3 * blk + 2);
    m.shared = false;
    m.nk = gate_up ? a.d / 64 : a.I / 64;
    m.ok = m.e >= 0 && m.e < a.E && m.rows >= 1 && m.rows <= kGemmBN && m.row0 >= 0 &&
           m.row0 + m.rows <= a.T * a.k;
  } else {
    const int j = it - s.n_routed;
    const int sblk = j / s.mt_s;
    m.mt = j % s.mt_s;
    m.e = 0;
    m.row0 = sblk * kGemmBN;
    m.rows = min(kGemmBN, a.T - m.row0);
    m.shared = true;
    m.nk = gate_up ? a.d / 64 : a.I_shared / 64;
    m.ok = true;
  }
  return m;
}

__device__ __forceinline__ int tile_n(int rows) { return max(16, (rows + 15) & ~15); }

// pipeline stages of an item of nk groups, kG groups a stage (the last may
// hold fewer)
template <int kG>
__device__ __forceinline__ int n_stages(int nk) { return (nk + kG - 1) / kG; }

// Eight 4-bit codes of one word in the interleaved order of the prepacked
// layout (code 2p in bits 4p, code 2p+1 in bits 4p+16) -> four f16x2 values of
// q*scale + bias, adjacent columns paired (low half = lower k).  A mask puts
// 1024 + q (codes in bits 0..3 and 16..19) or 1024 + 16 q (bits 4..7, 20..23)
// into an f16 pair; one fp16 FMA recovers q exactly, one more applies scale
// and bias.  fp16 carries 11 significant bits, so q*scale + bias is exact
// whenever it fits them (always when bias = -8*scale: |q-8| <= 8 adds at most
// 3 bits to the 8-bit bf16 scale); otherwise it is rounded once.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s2, uint32_t b2, uint32_t* out) {
  const uint32_t magic = 0x64006400u;  // f16 pair (1024, 1024)
  const uint32_t w8 = w >> 8;
  const uint32_t v0 = lop3_and_or(w, 0x000F000Fu, magic);    // 1024 + q: codes 0, 1
  const uint32_t v1 = lop3_and_or(w, 0x00F000F0u, magic);    // 1024 + 16 q: codes 2, 3
  const uint32_t v2 = lop3_and_or(w8, 0x000F000Fu, magic);   // codes 4, 5
  const uint32_t v3 = lop3_and_or(w8, 0x00F000F0u, magic);   // codes 6, 7
  const uint32_t one = 0x3C003C00u, minus_1024 = 0xE400E400u;      // f16 pairs (1, 1), (-1024, -1024)
  const uint32_t sixteenth = 0x2C002C00u, minus_64 = 0xD400D400u;  // (1/16, 1/16), (-64, -64)
  out[0] = f16x2_fma(f16x2_fma(v0, one, minus_1024), s2, b2);
  out[1] = f16x2_fma(f16x2_fma(v1, sixteenth, minus_64), s2, b2);
  out[2] = f16x2_fma(f16x2_fma(v2, one, minus_1024), s2, b2);
  out[3] = f16x2_fma(f16x2_fma(v3, sixteenth, minus_64), s2, b2);
}

// Sixteen 2-bit codes of one word in the interleaved order of the prepacked
// layout (code 2p in bits 2p, code 2p+1 in bits 2p+16) -> eight f16x2 values
// of q*scale + bias, adjacent columns paired.  A mask leaves pair p at bits 2p
// as the f16 pair 1024 + 4^p q, exact for p <= 4 (at most 1792); one fp16 FMA
// by 4^-p recovers q exactly, one more applies scale and bias.  Pairs 5..7
// take one shift first.
__device__ __forceinline__ void dequant_word2(uint32_t w, uint32_t s2, uint32_t b2, uint32_t* out) {
  const uint32_t magic = 0x64006400u;  // f16 pair (1024, 1024)
  // f16 pairs (4^-p, 4^-p) and (-1024 * 4^-p, ...) for p = 0..4
  constexpr uint32_t kScale[5] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u, 0x1C001C00u};
  constexpr uint32_t kShift[5] = {0xE400E400u, 0xDC00DC00u, 0xD400D400u, 0xCC00CC00u, 0xC400C400u};
  const uint32_t w10 = w >> 10;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int pp = p < 5 ? p : p - 5;
    const uint32_t v = lop3_and_or(p < 5 ? w : w10, 0x00030003u << (2 * pp), magic);
    out[p] = f16x2_fma(f16x2_fma(v, kScale[pp], kShift[pp]), s2, b2);
  }
}

// Sixteen 3-bit codes of one 16-column block (lo: its low two bits in the
// 2-bit interleaved order; hi: its high bits, pair p's at bits p and p+16)
// -> eight f16x2 values of q*scale + bias.  The masks leave the f16 pairs
// 1024 + 4^pp lo (pair p in place in lo, or in lo >> 10: pp = p or p - 5) and
// 1024 + 2^p hi; the first FMA turns the second into 4 hi - 1024 4^-pp, the
// second adds lo + 1024 4^-pp, so q = lo + 4 hi comes out exactly (every
// intermediate is an integer or a short binary fraction below 2048), and the
// third applies scale and bias.
__device__ __forceinline__ void dequant_word3(uint32_t lo, uint32_t hi, uint32_t s2, uint32_t b2, uint32_t* out) {
  const uint32_t magic = 0x64006400u;  // f16 pair (1024, 1024)
  constexpr uint32_t kScale[5] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u, 0x1C001C00u};  // 4^-pp
  // f16 pairs (4 * 2^-p, ...) and (-(4096 * 2^-p + 1024 * 4^-pp), ...) for p = 0..7
  constexpr uint32_t kHiScale[8] = {0x44004400u, 0x40004000u, 0x3C003C00u, 0x38003800u,
                                    0x34003400u, 0x30003000u, 0x2C002C00u, 0x28002800u};
  constexpr uint32_t kHiShift[8] = {0xED00ED00u, 0xE880E880u, 0xE440E440u, 0xE020E020u,
                                    0xDC10DC10u, 0xE480E480u, 0xDD00DD00u, 0xD600D600u};
  const uint32_t lo10 = lo >> 10;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int pp = p < 5 ? p : p - 5;
    const uint32_t vl = lop3_and_or(p < 5 ? lo : lo10, 0x00030003u << (2 * pp), magic);
    const uint32_t vh = lop3_and_or(hi, 0x00010001u << p, magic);
    const uint32_t t = f16x2_fma(vh, kHiScale[p], kHiShift[p]);
    out[p] = f16x2_fma(f16x2_fma(vl, kScale[pp], t), s2, b2);
  }
}

template <bool kGateUp, int kBits>
__global__ void __launch_bounds__(Cfg<kGateUp, kBits>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap q0_r, const __grid_constant__ CUtensorMap q1_r,
                    const __grid_constant__ CUtensorMap sb0_r, const __grid_constant__ CUtensorMap sb1_r,
                    const __grid_constant__ CUtensorMap q0_s, const __grid_constant__ CUtensorMap q1_s,
                    const __grid_constant__ CUtensorMap sb0_s, const __grid_constant__ CUtensorMap sb1_s,
                    const __grid_constant__ CUtensorMap act0, const __grid_constant__ CUtensorMap act1,
                    const __grid_constant__ CUtensorMap out_map, GemmArgs a) {
  using C = Cfg<kGateUp, kBits>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* epi_stage = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes + C::kEpiStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + C::kStages;
  uint64_t* a_full = empty + C::kStages;
  uint64_t* a_empty = a_full + C::kAStages;
  uint64_t* acc_full = a_empty + C::kAStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);  // the producer's expect_tx arrival; the bytes complete the phase
      mbar_init(&empty[i], C::kEmptyArrivals);
    }
    for (int i = 0; i < C::kAStages; ++i) {
      mbar_init(&a_full[i], C::kDqWarps);
      mbar_init(&a_empty[i], C::kAEmptyArrivals);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], C::kMmaIssuers);  // one commit per MMA issuer
      mbar_init(&acc_empty[i], C::kEpiWarps);
    }
    mbar_init(&done[0], 1);
    mbar_init(&done[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&q0_r);
    tma_prefetch_desc(&sb0_r);
    tma_prefetch_desc(&act0);
    if (kGateUp) {
      tma_prefetch_desc(&q1_r);
      tma_prefetch_desc(&sb1_r);
    }
  }
  if (warp == kMmaWarp0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();  // routing, X (and for the down GEMM, h) come from earlier kernels
  pdl_launch_dependents();

  Sched s;
  s.nb = *a.num_blocks;
  if (s.nb < 0 || s.nb > a.max_blocks) {
    if (threadIdx.x == 0) record_status(a.status, MOE_ERR_INVALID_ARG);
    s.nb = 0;
  }
  s.mt_r = kGateUp ? (a.I + kGemmBM - 1) / kGemmBM : (a.d + kGemmBM - 1) / kGemmBM;
  s.mt_s = kGateUp ? (a.I_shared + kGemmBM - 1) / kGemmBM : s.mt_r;
  s.nsb = a.I_shared > 0 ? (a.T + kGemmBN - 1) / kGemmBN : 0;
  s.n_routed = s.nb * s.mt_r;
  s.n_total = s.n_routed + s.nsb * s.mt_s;

  // one k-block's codes of one 128-row tile: 4- and 2-bit codes one 3-D box;
  // 3-bit codes (24 bytes a row, a line of 8-byte units [E*K/64][N*3]) two
  // boxes of 64 rows, `half` choosing one
  // one stage's codes of one 128-row tile from group eg on: 4- and 2-bit
  // codes one 3-D box of kG groups; 3-bit codes (24 bytes a row, a line of
  // 8-byte units [E*K/64][N*3]) two boxes of 64 rows per group.  Groups past
  // the item's last are read (the next expert's, or zeros past the tensor) and
  // then ignored.
  auto load_codes = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int mt, int eg) {
    if constexpr (kBits == 3) {
#pragma unroll
      for (int g = 0; g < C::kG; ++g)
#pragma unroll
        for (int half = 0; half < 2; ++half)
          tma_load_2d(dst + g * C::kQBytesG + half * (C::kQBytesG / 2), map, bar,
                      (mt * kGemmBM + half * (kGemmBM / 2)) * 3, eg + g);
    } else {
      tma_load_3d(dst, map, bar, 0, mt * kGemmBM, eg);
    }
  };
  auto fail = [&]() {
    record_status(a.status, MOE_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t used_mask = 0, last_parity = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < s.n_total && ok; it += gridDim.x) {
      const Item m = get_item(a, s, it, kGateUp);
      if (!m.ok) continue;
      const CUtensorMap* mq0 = m.shared ? &q0_s : &q0_r;
      const CUtensorMap* mq1 = m.shared ? &q1_s : &q1_r;
      const CUtensorMap* msb0 = m.shared ? &sb0_s : &sb0_r;
      const CUtensorMap* msb1 = m.shared ? &sb1_s : &sb1_r;
      // token tile: kGemmBN rows of the activation tensor from the item's
      // first row (rows past the item belong to the next item or lie past the
      // end of the tensor and are zero-filled; their MMA columns are ignored)
      const CUtensorMap* mb = (!kGateUp && m.shared) ? &act1 : &act0;
      const int brow = (kGateUp && m.shared) ? a.T * a.k + m.row0 : m.row0;
      if (lane == 0) {
        for (int ks = 0; ks < n_stages<C::kG>(m.nk); ++ks) {
          const int kb = ks * C::kG;  // first group of the stage
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          uint8_t* st = stages + stage * C::kStageBytes;
          uint8_t* q_tile = st + C::kBBytes;
          uint8_t* sb_tile = q_tile + C::kMats * C::kQBytes;
          const int eg = m.e * m.nk + kb;
          mbar_arrive_expect_tx(&full[stage], C::kStageTxBytes);
#pragma unroll
          for (int g = 0; g < C::kG; ++g)  // columns past the tensor's last are zeros
            tma_load_2d(st + g * C::kBBoxBytes, mb, &full[stage], (kb + g) * 64, brow);
          load_codes(q_tile, mq0, &full[stage], m.mt, eg);
          tma_load_3d(sb_tile, msb0, &full[stage], m.mt * kGemmBM, kb, m.e);
          if (kGateUp) {
            load_codes(q_tile + C::kQBytes, mq1, &full[stage], m.mt, eg);
            tma_load_3d(sb_tile + C::kSBBytes, msb1, &full[stage], m.mt * kGemmBM, kb, m.e);
          }
          used_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    // never leave while a load into this CTA's shared memory may be in flight
    if (lane == 0) {
      for (int i = 0; i < C::kStages; ++i)
        if ((used_mask >> i) & 1u) {
          if (!mbar_wait(&full[i], (last_parity >> i) & 1u, nullptr)) record_status(a.status, MOE_ERR_TIMEOUT);
        }
    }
    __syncwarp();
  } else if (warp == kMmaWarp0 + 1 && C::kMmaIssuers == 1) {
    // the down GEMM's second MMA warp idles
  } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
    // ------------------------------------------------------------ MMA issuers
    // gate/up: issuer 0 multiplies the gate tile, issuer 1 the up tile, both
    // over every stage.  down: one issuer.
    const int who = warp - kMmaWarp0;
    // shared-memory addresses stay below 2^18, so the descriptor's 14-bit
    // address field never carries into its neighbours
    const uint64_t b_desc0 = smem_desc_sw128_kmajor(smem_u32(stages));
    int stage = 0, astage = 0, accb = 0;
    uint32_t aphase = 0, accphase = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < s.n_total && ok; it += gridDim.x) {
      const Item m = get_item(a, s, it, kGateUp);
      if (!m.ok) continue;
      const int bn = tile_n(m.rows);
      const uint32_t idesc = idesc_f16_f32(kGemmBM, bn);
      if (!mbar_wait(&acc_empty[accb], accphase ^ 1, abort_flag)) {
        fail();
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + accb * C::kAccBufCols + who * kGemmBN;
      bool first = true;
      for (int ks = 0; ks < n_stages<C::kG>(m.nk); ++ks) {
        // a_full completes only after every dequantisation warp has seen
        // full[stage] complete (the stage's token tile has landed) and
        // arrived with release semantics, so waiting on a_full alone orders
        // these MMAs after the tile's TMA writes as well
        if (!mbar_wait(&a_full[astage], aphase, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          // the four K = 16 slices of each group: 32 bytes apart in the
          // group's swizzled token box (2 in the descriptor's address
          // field), 8 columns apart in the A stage; a group past the item's
          // last multiplies zero weights by zero tokens
          const uint64_t bd = b_desc0 + static_cast<uint64_t>(stage * (C::kStageBytes >> 4));
          const uint32_t a0 = tmem + C::kABase + astage * C::kACols + (kGateUp ? who * 32 * C::kG : 0);
#pragma unroll
          for (int g = 0; g < C::kG; ++g) {
            const uint64_t bg = bd + static_cast<uint64_t>(g * (C::kBBoxBytes >> 4));
            tc_mma_ts(d, a0 + 32 * g, bg, idesc, (first && g == 0) ? 0u : 1u);
            tc_mma_ts(d, a0 + 32 * g + 8, bg + 2, idesc, 1u);
            tc_mma_ts(d, a0 + 32 * g + 16, bg + 4, idesc, 1u);
            tc_mma_ts(d, a0 + 32 * g + 24, bg + 6, idesc, 1u);
          }
          tc_commit(&empty[stage]);
          tc_commit(&a_empty[astage]);
        }
        __syncwarp();
        first = false;
        if (++stage == C::kStages) stage = 0;
        if (++astage == C::kAStages) {
          astage = 0;
          aphase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&acc_full[accb]);  // arrives at once if this issuer had no k-block
      __syncwarp();
      if (++accb == C::kAccBufs) {
        accb = 0;
        accphase ^= 1;
      }
    }
    // all MMAs issued by this thread have completed before TMEM is released
    if (lane == 0) {
      tc_commit(&done[who]);
      if (!mbar_wait(&done[who], 0, nullptr)) record_status(a.status, MOE_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= C::kDqWarp0) {
    // ------------------------------------------------------------ dequantisation
    const int lanegrp = warp & 3;
    const int row = lanegrp * 32 + lane;  // weight row inside the tile = TMEM lane
    const int mat = (warp - C::kDqWarp0) >> 2;
    const int swz = (row >> 2) & 1;
    int stage = 0, astage = 0;
    uint32_t phase = 0, aphase = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < s.n_total && ok; it += gridDim.x) {
      const Item m = get_item(a, s, it, kGateUp);
      if (!m.ok) continue;
      for (int ks = 0; ks < n_stages<C::kG>(m.nk); ++ks) {
        // every warp waits for itself: no warp holds the others back, and the
        // warps drift apart, so their bursts do not all compete for issue
        // slots with the MMA issuer at once
        if (!mbar_wait(&full[stage], phase, abort_flag) || !mbar_wait(&a_empty[astage], aphase ^ 1, abort_flag)) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = stages + stage * C::kStageBytes;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(lanegrp * 32) << 16) + C::kABase + astage * C::kACols +
                               mat * 32 * C::kG;
        // every code word and group parameter of this row in the stage is
        // loaded before any is used, so that the loads' latency is paid once
        // (the TMEM stores below are ordered memory operations, which the
        // compiler does not move loads across)
        const uint8_t* q_base = st + C::kBBytes + mat * C::kQBytes;
        const uint8_t* sb_base = st + C::kBBytes + C::kMats * C::kQBytes + mat * C::kSBBytes + row * 4;
        constexpr int kRaw = 2 * kBits;  // code words of one row and group
        uint32_t raw[C::kG][kRaw], sbv[C::kG];
#pragma unroll
        for (int g = 0; g < C::kG; ++g) {
          const uint8_t* q_tile = q_base + g * C::kQBytesG;
          sbv[g] = *reinterpret_cast<const uint32_t*>(sb_base + g * C::kSBBytesG);
          if constexpr (kBits == 4) {
            // the row's 32 code bytes are two 16-byte halves, swapped in rows
            // where the 32-byte swizzle flips bit 4 of the address; half h
            // holds words 4h .. 4h+3 = columns 32h .. 32h+31
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 w = *reinterpret_cast<const uint4*>(q_tile + row * 32 + ((h ^ swz) << 4));
              raw[g][4 * h + 0] = w.x;
              raw[g][4 * h + 1] = w.y;
              raw[g][4 * h + 2] = w.z;
              raw[g][4 * h + 3] = w.w;
            }
          } else if constexpr (kBits == 3) {
            // the row's 24 code bytes: low-bit words j = 0..3 (columns 16j .. 16j+15), then the high-bit
            // words of blocks 0, 1 and 2, 3 (block 2i+1 in the upper byte of each half)
            const uint2* rp = reinterpret_cast<const uint2*>(q_tile + row * 24);
            const uint2 l01 = rp[0], l23 = rp[1], hh = rp[2];
            raw[g][0] = l01.x;
            raw[g][1] = l01.y;
            raw[g][2] = l23.x;
            raw[g][3] = l23.y;
            raw[g][4] = hh.x;
            raw[g][5] = hh.y;
          } else {
            // the row's 16 code bytes: words j = 0..3 hold columns 16j .. 16j+15
            const uint4 w = *reinterpret_cast<const uint4*>(q_tile + row * 16);
            raw[g][0] = w.x;
            raw[g][1] = w.y;
            raw[g][2] = w.z;
            raw[g][3] = w.w;
          }
        }
#pragma unroll
        for (int g = 0; g < C::kG; ++g) {
          const uint32_t tg = taddr + 32 * g;
          if (g > 0 && ks * C::kG + g >= m.nk) {
            // past the item's last group: zero weights (the token columns there are zeros too, but the codes
            // and parameters read for them belong to another matrix)
            uint32_t z[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) z[c] = 0u;
            tmem_st16(tg, z);
            tmem_st16(tg + 16, z);
            continue;
          }
          const float sf = __uint_as_float(sbv[g] << 16);  // bf16 -> fp32 is exact
          const float bf = __uint_as_float(sbv[g] & 0xFFFF0000u);
          const uint32_t s2 = f32x2_to_f16x2(sf, sf);
          const uint32_t b2 = f32x2_to_f16x2(bf, bf);
          uint32_t v[16];
          if constexpr (kBits == 4) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              dequant_word(raw[g][4 * h + 0], s2, b2, v + 0);
              dequant_word(raw[g][4 * h + 1], s2, b2, v + 4);
              dequant_word(raw[g][4 * h + 2], s2, b2, v + 8);
              dequant_word(raw[g][4 * h + 3], s2, b2, v + 12);
              tmem_st16(tg + h * 16, v);
            }
          } else if constexpr (kBits == 3) {
            dequant_word3(raw[g][0], raw[g][4], s2, b2, v + 0);
            dequant_word3(raw[g][1], raw[g][4] >> 8, s2, b2, v + 8);
            tmem_st16(tg, v);
            dequant_word3(raw[g][2], raw[g][5], s2, b2, v + 0);
            dequant_word3(raw[g][3], raw[g][5] >> 8, s2, b2, v + 8);
            tmem_st16(tg + 16, v);
          } else {
            dequant_word2(raw[g][0], s2, b2, v + 0);
            dequant_word2(raw[g][1], s2, b2, v + 8);
            tmem_st16(tg, v);
            dequant_word2(raw[g][2], s2, b2, v + 0);
            dequant_word2(raw[g][3], s2, b2, v + 8);
            tmem_st16(tg + 16, v);
          }
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[stage]);
          mbar_arrive(&a_full[astage]);
        }
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++astage == C::kAStages) {
          astage = 0;
          aphase ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ep = warp - kEpiWarp0;
    const int lanegrp = warp & 3;
    const int colpart = ep >> 2;  // this warp handles columns [colpart * kEpiCols, (colpart + 1) * kEpiCols)
    const int row = lanegrp * 32 + lane;
    int accb = 0;
    uint32_t accphase = 0;
    uint32_t nstore = 0;  // TMA stores issued by this warp (down GEMM), alternating its two staging buffers
    for (int it = blockIdx.x; it < s.n_total; it += gridDim.x) {
      const Item m = get_item(a, s, it, kGateUp);
      if (!m.ok) {
        if (lane == 0) record_status(a.status, MOE_ERR_INVALID_ARG);
        continue;
      }
      const int bn = tile_n(m.rows);
      const int c_begin = colpart * C::kEpiCols;
      const int c_end = min(bn, c_begin + C::kEpiCols);
      bool bad = false;
      if (ep == 0) {
        bad = !mbar_wait(&acc_full[accb], accphase, abort_flag);
        if (bad && lane == 0) fail();
      }
      if (bar_sync_or(kBarEpilogue, C::kEpiWarps * 32, bad)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(lanegrp * 32) << 16) + accb * C::kAccBufCols;
      const int n = m.mt * kGemmBM + row;
      if constexpr (kGateUp) {
        // h = SiLU(gate) * up, rounded to fp16 (the down GEMM's operand);
        // rows of h follow the item's rows (permuted order, or token order for
        // the shared expert)
        const int Icur = m.shared ? a.I_shared : a.I;
        uint16_t* H = (m.shared ? a.h_shared : a.h_routed) + static_cast<size_t>(m.row0) * Icur + n;
        const int c_valid = min(c_end, m.rows);
        bool range_ok = true;
        // 16 columns of gate and up per TMEM round trip (the column ranges
        // are multiples of 16: kEpiCols and the tile width both are)
        for (int c0 = c_begin; c0 < c_end; c0 += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(tbase + c0, g);
          tmem_ld16(tbase + kGemmBN + c0, u);
          tc_wait_ld();
          if (n < Icur) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              if (c0 + c < c_valid) {
                // SiLU(g) u = (g/2) u (1 + tanh(g/2)), the logistic function
                // written through tanh: one special-function instruction
                // instead of an exponential and a reciprocal.  tanh.approx's
                // absolute error (about 2^-11) puts at most about |g u| 2^-12 on
                // h, the order of h's own rounding to fp16.
                const float t = 0.5f * __uint_as_float(g[c]);
                const float pv = t * __uint_as_float(u[c]);
                float th;
                asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(t));
                const float h = fmaf(pv, th, pv);
                range_ok &= fabsf(h) <= 65504.0f;
                H[static_cast<size_t>(c0 + c) * Icur] = __half_as_ushort(__float2half_rn(h));
              }
            }
          }
        }
        if (!range_ok) record_status(a.status, MOE_ERR_UNSUPPORTED);
      } else {
        // expert output rows: routed items in permuted order (row p of the
        // routing), shared-expert items after them in token order; the combine
        // kernel applies the routing weights and gathers rows back to tokens.
        // A full round of 16 tokens goes out as one TMA store of the warp's 32
        // rows, staged in shared memory; a partial round (the item's last
        // rows) as plain stores, so that no row past the item is written.
        const size_t row_base = (m.shared ? static_cast<size_t>(a.T) * a.k : 0) + m.row0;
        const int n0 = m.mt * kGemmBM + lanegrp * 32;
        const int c_valid = min(c_end, m.rows);
        for (int c0 = c_begin; c0 < c_end; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tbase + c0, v);
          tc_wait_ld();
          if (c_valid - c0 >= 16) {
            float* buf = epi_stage + (ep * 2 + (nstore & 1u)) * C::kEpiBufFloats;
            if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 16; ++c) buf[c * 32 + lane] = __uint_as_float(v[c]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&out_map, buf, n0, static_cast<int>(row_base + c0));
              bulk_commit_group();
            }
            ++nstore;
          } else if (n < a.d) {
            float* Yp = a.ypart + (row_base + c0) * a.d + n;
#pragma unroll
            for (int c = 0; c < 16; ++c)
              if (c0 + c < c_valid) Yp[static_cast<size_t>(c) * a.d] = __uint_as_float(v[c]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[accb]);
      if (++accb == C::kAccBufs) {
        accb = 0;
        accphase ^= 1;
      }
    }
    if (!kGateUp && lane == 0) bulk_wait_group_all();  // the staged stores are done before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp0) tmem_dealloc(tmem, kTmemCols);
}

// The gate/up GEMM's token operand: fp16 rows of X in the routing's permuted
// order (row p = X[perm[p] / k]), followed by the T rows of X in token order
// when there is a shared expert.  Values outside the fp16 range are recorded
// as MOE_ERR_UNSUPPORTED.  One warp per row: every lane's 16-byte pieces of
// the row are loaded before any is converted.
constexpr int kGatherThreads = 256;
constexpr int kGatherU = 8;  // 16-byte pieces per lane in flight (a 2048-wide row in one round)
__global__ void __launch_bounds__(kGatherThreads)
    x_gather_kernel(const uint16_t* __restrict__ X, const int32_t* __restrict__ perm, int T, int d, int k, int rows,
                    uint16_t* __restrict__ Xg, uint32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int A = T * k;
  const int d8 = d / 8;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (kGatherThreads / 32);
  // |x| <= 65504 (the fp16 range) for a bf16 x is (bits & 0x7FFF) <= 0x477F,
  // 0x477F being the largest finite bf16 below 65504 (NaN and infinity lie
  // above it): a running maximum of both halves of every word, checked once
  uint32_t amax = 0;
  bool idx_ok = true;
  for (int r = blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    const int t = r < A ? __ldg(perm + r) / k : r - A;
    if (t < 0 || t >= T) {
      idx_ok = false;
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(X) + static_cast<size_t>(t) * d8;
    uint4* dst = reinterpret_cast<uint4*>(Xg) + static_cast<size_t>(r) * d8;
    for (int c0 = lane; c0 < d8; c0 += 32 * kGatherU) {
      uint4 v[kGatherU];
#pragma unroll
      for (int u = 0; u < kGatherU; ++u)
        if (c0 + 32 * u < d8) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kGatherU; ++u) {
        if (c0 + 32 * u >= d8) continue;
        const uint32_t in[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          amax = __vmaxu2(amax, in[j] & 0x7FFF7FFFu);
          out[j] = f32x2_to_f16x2(__uint_as_float(in[j] << 16), __uint_as_float(in[j] & 0xFFFF0000u));
        }
        dst[c0 + 32 * u] = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
  }
  if ((amax & 0xFFFFu) > 0x477Fu || (amax >> 16) > 0x477Fu) record_status(status, MOE_ERR_UNSUPPORTED);
  if (!idx_ok) record_status(status, MOE_ERR_INVALID_ARG);
}

// Y[t] = bf16( sum_j w[t][j] * yexp[inv_perm[t*k + j]] + yexp[A + t] ): the
// weighted top-k combine plus the shared expert, summed in slot order.  One
// CTA per token (grid-stride); each thread owns float4 columns and issues the
// loads of every slot before it sums them in slot order.
constexpr int kCombineThreads = 256;
constexpr int kCombineSlots = 8;  // slots whose rows are in flight together
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float* __restrict__ ypart, const int32_t* __restrict__ inv_perm,
                   const float* __restrict__ w, int T, int d, int k, int has_shared, uint16_t* __restrict__ Y,
                   uint32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t A = static_cast<size_t>(T) * k;
  const int d4 = d / 4;
  bool ok = true;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    for (int c = threadIdx.x; c < d4; c += kCombineThreads) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = 0; j0 < k; j0 += kCombineSlots) {
        float4 v[kCombineSlots];
        float wj[kCombineSlots];
        bool in[kCombineSlots];
#pragma unroll
        for (int u = 0; u < kCombineSlots; ++u) {
          const int j = j0 + u;
          in[u] = false;
          if (j < k) {
            const int p = __ldg(inv_perm + static_cast<size_t>(t) * k + j);
            wj[u] = __ldg(w + static_cast<size_t>(t) * k + j);
            if (p < 0 || static_cast<size_t>(p) >= A) {
              ok = false;
            } else {
              in[u] = true;
              v[u] = *reinterpret_cast<const float4*>(ypart + static_cast<size_t>(p) * d + 4 * c);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kCombineSlots; ++u) {
          if (!in[u]) continue;
          acc.x = fmaf(wj[u], v[u].x, acc.x);
          acc.y = fmaf(wj[u], v[u].y, acc.y);
          acc.z = fmaf(wj[u], v[u].z, acc.z);
          acc.w = fmaf(wj[u], v[u].w, acc.w);
        }
      }
      if (has_shared) {
        const float4 v = *reinterpret_cast<const float4*>(ypart + (A + t) * d + 4 * c);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.x))) |
                          (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.y))) << 16);
      const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.z))) |
                          (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.w))) << 16);
      *reinterpret_cast<uint2*>(Y + static_cast<size_t>(t) * d + 4 * c) = make_uint2(lo, hi);
    }
  }
  if (!ok) record_status(status, MOE_ERR_INVALID_ARG);
}

template <int kBits>
cudaError_t launch_gemm_t(const GemmArgs& a, const GemmMaps* routed, const GemmMaps* shared,
                          const GemmActMaps* act, cudaStream_t stream, bool pdl) {
  using CG = Cfg<true, kBits>;
  using CD = Cfg<false, kBits>;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(moe_gemm_kernel<true, kBits>), CG::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = set_max_dynamic_smem(reinterpret_cast<const void*>(moe_gemm_kernel<false, kBits>), CD::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  const GemmMaps* sh = shared ? shared : routed;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(a.num_sms);

  {
    cudaLaunchConfig_t c2 = cfg;
    const int rows = a.T * a.k + (a.I_shared > 0 ? a.T : 0);
    constexpr int kRowsPerCta = kGatherThreads / 32;
    c2.gridDim = dim3(max(1, min((rows + kRowsPerCta - 1) / kRowsPerCta, a.num_sms * 16)));
    c2.blockDim = dim3(kGatherThreads);
    c2.dynamicSmemBytes = 0;
    timer_begin(kKXGather, stream);
    cudaError_t e = cudaLaunchKernelEx(&c2, x_gather_kernel, a.X, a.perm, a.T, a.d, a.k, rows, a.Xh, a.status);
    timer_end(kKXGather, stream);
    if (e != cudaSuccess) return e;
  }
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.dynamicSmemBytes = CG::kSmemBytes;
  cfg.blockDim = dim3(CG::kThreads);
  timer_begin(kKGemmGateUp, stream);
  cudaError_t err = cudaLaunchKernelEx(&cfg, moe_gemm_kernel<true, kBits>, routed->q_gate, routed->q_up, routed->sb_gate,
                                       routed->sb_up, sh->q_gate, sh->q_up, sh->sb_gate, sh->sb_up, act->x, act->x,
                                       act->ypart, a);
  timer_end(kKGemmGateUp, stream);
  if (err != cudaSuccess) return err;

  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.dynamicSmemBytes = CD::kSmemBytes;
  cfg.blockDim = dim3(CD::kThreads);
  timer_begin(kKGemmDown, stream);
  err = cudaLaunchKernelEx(&cfg, moe_gemm_kernel<false, kBits>, routed->q_down, routed->q_down, routed->sb_down,
                           routed->sb_down, sh->q_down, sh->q_down, sh->sb_down, sh->sb_down, act->h_routed,
                           act->h_shared, act->ypart, a);
  timer_end(kKGemmDown, stream);
  if (err != cudaSuccess) return err;

  cfg.gridDim = dim3(max(1, min(a.T, a.num_sms * 8)));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  timer_begin(kKCombine, stream);
  err = cudaLaunchKernelEx(&cfg, combine_kernel, static_cast<const float*>(a.ypart), a.inv_perm, a.w, a.T, a.d, a.k,
                           a.I_shared > 0 ? 1 : 0, a.Y, a.status);
  timer_end(kKCombine, stream);
  return err;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, const GemmMaps* routed, const GemmMaps* shared, const GemmActMaps* act,
                        cudaStream_t stream, bool pdl) {
  if (a.bits == 2) return launch_gemm_t<2>(a, routed, shared, act, stream, pdl);
  if (a.bits == 3) return launch_gemm_t<3>(a, routed, shared, act, stream, pdl);
  if (a.bits == 4) return launch_gemm_t<4>(a, routed, shared, act, stream, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace bm
