// Prefill path: grouped expert GEMMs on the 5th-generation tensor cores with
// the 4-bit dequantisation fused in ("Perplexity's Lily Beats MLX-LM on
// MacBook M5", section "Prefill: keep routing on the GPU, dequantize in
// flight": the grouped GEMM dequantises one small tile at a time on chip,
// accumulates in FP32, writes bf16 and never materialises the expanded
// weights; the expert input projections are fused with the gate activation and
// the output projection with the routing scores and the shared expert).
//
// Operands are fp16 (the pages' Metal kernels use bf16): fp16 holds the
// dequantised weights of this format exactly and rounds h and X 8x more finely,
// at the same tensor-core rate; X is converted once per call.
//
// sm_103a design ("swap AB"): the weights are the M = 128 operand and an
// expert's tokens the N operand (16..128, a multiple of 16), so an expert with
// few tokens still streams its weight tile exactly once.  The dequantised
// weight tile never touches shared memory: dequantisation warps turn the TMA-
// loaded codes into fp16 and store them with tcgen05.st straight into tensor
// memory, where tcgen05.mma reads them as its A operand; shared memory carries
// only the packed codes, the group parameters and the token tile (TMA gather4
// of the expert's token rows).  Accumulators live in tensor memory.
//
// Roles (14 warps, one persistent CTA per SM):
//   warps 0-7   dequantise codes -> fp16 A tiles in TMEM
//   warps 8-11  epilogue: TMEM -> registers -> SwiGLU (gate/up) or weighted
//               scatter of expert outputs (down)
//   warp 12     TMA producer (codes, group parameters, token rows)
//   warp 13     MMA issuer (one lane)
// Synchronisation is by mbarriers; every wait is bounded (2 s) and records
// MOE_ERR_TIMEOUT instead of hanging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bm {

namespace {

constexpr int kThreads = 448;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint32_t kTmemCols = 512;

template <bool kGateUp>
struct Cfg {
  static constexpr int kMats = kGateUp ? 2 : 1;
  static constexpr int kStages = kGateUp ? 6 : 8;
  static constexpr int kAStages = kGateUp ? 4 : 8;
  static constexpr int kACols = 32 * kMats;  // 64 fp16 per lane per matrix = 32 columns
  static constexpr int kAccCols = kMats * kGemmBN;
  static constexpr int kAccBufs = kGateUp ? 1 : 2;
  static constexpr int kABase = kAccBufs * kAccCols;
  static_assert(kABase + kAStages * kACols <= static_cast<int>(kTmemCols), "TMEM budget");
  static constexpr int kBBytes = kGemmBN * 128;  // token tile: up to 128 rows x 64 fp16 (128-byte swizzle)
  static constexpr int kQBytes = kGemmBM * 32;   // 128 rows x 8 code words (32-byte swizzle)
  static constexpr int kSBBytes = kGemmBM * 4;
  static constexpr int kStageBytes = ((kBBytes + kMats * (kQBytes + kSBBytes)) + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*barriers etc.*/ + 1024 /*align*/;
};

struct Item {
  int e, row0, rows, mt, nk;
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

// Eight 4-bit codes (one word, k ascending from the low nibble) -> four f16x2
// values of q*scale + bias, adjacent columns paired (low half = lower k).
// fp16 carries 11 significant bits, so q*scale + bias is exact whenever it fits
// them (always when bias = -8*scale: |q-8| <= 8 adds at most 3 bits to the
// 8-bit bf16 scale); otherwise it is rounded once.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s2, uint32_t b2, uint32_t* out) {
  const uint32_t w4 = w >> 4;
  const uint32_t magic = 0x64006400u;      // f16 pair (1024, 1024): a code in the low mantissa bits reads 1024 + q
  const uint32_t one = 0x3C003C00u;        // f16 pair (1, 1)
  const uint32_t minus_magic = 0xE400E400u;  // f16 pair (-1024, -1024)
  const uint32_t sel[4] = {0x4400u, 0x5511u, 0x6622u, 0x7733u};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t t = prmt(w, w4, sel[m]);                 // low nibbles: byte 0 = q_2m, byte 2 = q_2m+1
    const uint32_t v = lop3_and_or(t, 0x000F000Fu, magic);  // (1024 + q_2m, 1024 + q_2m+1)
    const uint32_t q = f16x2_fma(v, one, minus_magic);      // (q_2m, q_2m+1), exact
    out[m] = f16x2_fma(q, s2, b2);                          // q*scale + bias, one rounding
  }
}

template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap q0_r, const __grid_constant__ CUtensorMap q1_r,
                    const __grid_constant__ CUtensorMap sb0_r, const __grid_constant__ CUtensorMap sb1_r,
                    const __grid_constant__ CUtensorMap q0_s, const __grid_constant__ CUtensorMap q1_s,
                    const __grid_constant__ CUtensorMap sb0_s, const __grid_constant__ CUtensorMap sb1_s,
                    const __grid_constant__ CUtensorMap act_r, const __grid_constant__ CUtensorMap act_s,
                    GemmArgs a) {
  using C = Cfg<kGateUp>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + C::kStages;
  uint64_t* a_full = empty + C::kStages;
  uint64_t* a_empty = a_full + C::kAStages;
  uint64_t* acc_full = a_empty + C::kAStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 8 + 1);  // 8 dequantisation warps + the MMA commit
    }
    for (int i = 0; i < C::kAStages; ++i) {
      mbar_init(&a_full[i], 8);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&q0_r);
    tma_prefetch_desc(&sb0_r);
    tma_prefetch_desc(&act_r);
    if (kGateUp) {
      tma_prefetch_desc(&q1_r);
      tma_prefetch_desc(&sb1_r);
    }
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();  // routing and (for the down GEMM) h come from earlier kernels
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
      const int bn = tile_n(m.rows);
      const CUtensorMap* mq0 = m.shared ? &q0_s : &q0_r;
      const CUtensorMap* mq1 = m.shared ? &q1_s : &q1_r;
      const CUtensorMap* msb0 = m.shared ? &sb0_s : &sb0_r;
      const CUtensorMap* msb1 = m.shared ? &sb1_s : &sb1_r;
      const CUtensorMap* mact = m.shared ? &act_s : &act_r;
      // Token rows of the tile, loaded once per item: lane g owns rows 4g..4g+3
      // (the gather coordinates; rows past the tile read row T, out of range,
      // which TMA zero-fills).
      int tok[4] = {a.T, a.T, a.T, a.T};
      if (kGateUp) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int p = lane * 4 + i;
          if (p < m.rows) tok[i] = m.shared ? m.row0 + p : __ldg(a.perm + m.row0 + p) / a.k;
        }
      }
      const uint32_t bytes = C::kMats * (C::kQBytes + C::kSBBytes) + bn * 128;
      for (int kb = 0; kb < m.nk && ok; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        uint8_t* st = stages + stage * C::kStageBytes;
        uint8_t* b_tile = st;
        uint8_t* q_tile = st + C::kBBytes;
        uint8_t* sb_tile = q_tile + C::kMats * C::kQBytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_3d(q_tile, mq0, &full[stage], kb * 8, m.mt * kGemmBM, m.e);
          tma_load_3d(sb_tile, msb0, &full[stage], m.mt * kGemmBM, kb, m.e);
          if (kGateUp) {
            tma_load_3d(q_tile + C::kQBytes, mq1, &full[stage], kb * 8, m.mt * kGemmBM, m.e);
            tma_load_3d(sb_tile + C::kSBBytes, msb1, &full[stage], m.mt * kGemmBM, kb, m.e);
          }
          used_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        }
        __syncwarp();  // the expected byte count is registered before any row load can complete
        if (kGateUp) {
          if (lane < bn / 4)
            tma_gather4(b_tile + lane * 512, mact, &full[stage], kb * 64, tok[0], tok[1], tok[2], tok[3]);
        } else {
          if (lane < bn / 16) tma_load_2d(b_tile + lane * 2048, mact, &full[stage], kb * 64, m.row0 + lane * 16);
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // never leave while a load into this CTA's shared memory may be in flight
    if (lane == 0) {
      for (int i = 0; i < C::kStages; ++i)
        if ((used_mask >> i) & 1u) {
          if (!mbar_wait(&full[i], (last_parity >> i) & 1u, nullptr)) record_status(a.status, MOE_ERR_TIMEOUT);
        }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0, astage = 0, accb = 0;
    uint32_t phase = 0, aphase = 0, accphase = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < s.n_total && ok; it += gridDim.x) {
      const Item m = get_item(a, s, it, kGateUp);
      if (!m.ok) continue;
      const int bn = tile_n(m.rows);
      const uint32_t idesc = idesc_f16_f32(kGemmBM, bn);
      const int ab = kGateUp ? 0 : accb;
      if (!mbar_wait(&acc_empty[ab], accphase ^ 1, abort_flag)) {
        fail();
        break;
      }
      tc_fence_after();
      const uint32_t d0 = tmem + ab * C::kAccCols;
      for (int kb = 0; kb < m.nk; ++kb) {
        if (!mbar_wait(&a_full[astage], aphase, abort_flag) || !mbar_wait(&full[stage], phase, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t b_addr = smem_u32(stages + stage * C::kStageBytes);
          const uint32_t a0 = tmem + C::kABase + astage * C::kACols;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = smem_desc_sw128_kmajor(b_addr + kk * 32);
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            tc_mma_ts(d0, a0 + kk * 8, bdesc, idesc, acc);
            if (kGateUp) tc_mma_ts(d0 + kGemmBN, a0 + 32 + kk * 8, bdesc, idesc, acc);
          }
          tc_commit(&empty[stage]);
          tc_commit(&a_empty[astage]);
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++astage == C::kAStages) {
          astage = 0;
          aphase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&acc_full[ab]);
      __syncwarp();
      if (kGateUp) {
        accphase ^= 1;
      } else if (++accb == 2) {
        accb = 0;
        accphase ^= 1;
      }
    }
    // all MMAs issued by this thread have completed before TMEM is released
    if (lane == 0) {
      tc_commit(done);
      if (!mbar_wait(done, 0, nullptr)) record_status(a.status, MOE_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ dequantisation
    const int lanegrp = warp & 3;
    const int row = lanegrp * 32 + lane;             // weight row inside the tile = TMEM lane
    const int mat = kGateUp ? (warp >> 2) : 0;       // gate/up: which matrix
    const int half = warp >> 2;                      // down: which 32 columns of the group
    int stage = 0, astage = 0;
    uint32_t phase = 0, aphase = 0;
    bool ok = true;
    const int swz = (row >> 2) & 1;
    for (int it = blockIdx.x; it < s.n_total && ok; it += gridDim.x) {
      const Item m = get_item(a, s, it, kGateUp);
      if (!m.ok) continue;
      for (int kb = 0; kb < m.nk; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag) || !mbar_wait(&a_empty[astage], aphase ^ 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = stages + stage * C::kStageBytes;
        const uint8_t* q_tile = st + C::kBBytes + mat * C::kQBytes;
        const uint32_t sbv =
            *reinterpret_cast<const uint32_t*>(st + C::kBBytes + C::kMats * C::kQBytes + mat * C::kSBBytes + row * 4);
        const float sf = __uint_as_float(sbv << 16);          // bf16 -> fp32 is exact
        const float bf = __uint_as_float(sbv & 0xFFFF0000u);
        const uint32_t s2 = f32x2_to_f16x2(sf, sf);
        const uint32_t b2 = f32x2_to_f16x2(bf, bf);
        const uint32_t taddr = tmem + (static_cast<uint32_t>(lanegrp * 32) << 16) + C::kABase + astage * C::kACols;
        if constexpr (kGateUp) {
          const uint4 wa = *reinterpret_cast<const uint4*>(q_tile + row * 32 + ((0 ^ swz) * 16));
          const uint4 wb = *reinterpret_cast<const uint4*>(q_tile + row * 32 + ((1 ^ swz) * 16));
          uint32_t v[16];
          dequant_word(wa.x, s2, b2, v + 0);
          dequant_word(wa.y, s2, b2, v + 4);
          dequant_word(wa.z, s2, b2, v + 8);
          dequant_word(wa.w, s2, b2, v + 12);
          tmem_st16(taddr + mat * 32, v);
          dequant_word(wb.x, s2, b2, v + 0);
          dequant_word(wb.y, s2, b2, v + 4);
          dequant_word(wb.z, s2, b2, v + 8);
          dequant_word(wb.w, s2, b2, v + 12);
          tmem_st16(taddr + mat * 32 + 16, v);
        } else {
          const uint4 wv = *reinterpret_cast<const uint4*>(q_tile + row * 32 + ((half ^ swz) * 16));
          uint32_t v[16];
          dequant_word(wv.x, s2, b2, v + 0);
          dequant_word(wv.y, s2, b2, v + 4);
          dequant_word(wv.z, s2, b2, v + 8);
          dequant_word(wv.w, s2, b2, v + 12);
          tmem_st16(taddr + half * 16, v);
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
    const int lanegrp = warp & 3;
    const int row = lanegrp * 32 + lane;
    int accb = 0;
    uint32_t accphase = 0;
    for (int it = blockIdx.x; it < s.n_total; it += gridDim.x) {
      const Item m = get_item(a, s, it, kGateUp);
      if (!m.ok) {
        if (lane == 0) record_status(a.status, MOE_ERR_INVALID_ARG);
        continue;
      }
      const int bn = tile_n(m.rows);
      const int ab = kGateUp ? 0 : accb;
      if (!mbar_wait(&acc_full[ab], accphase, abort_flag)) {
        fail();
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(lanegrp * 32) << 16) + ab * C::kAccCols;
      const int n = m.mt * kGemmBM + row;
      if (kGateUp) {
        const int Icur = m.shared ? a.I_shared : a.I;
        uint16_t* H = m.shared ? a.h_shared : a.h_routed;
        for (int c0 = 0; c0 < bn; c0 += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(tbase + c0, g);
          tmem_ld16(tbase + kGemmBN + c0, u);
          tc_wait_ld();
          if (n < Icur) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              if (c0 + c < m.rows) {
                const float gv = __uint_as_float(g[c]);
                const float uv = __uint_as_float(u[c]);
                const float h = gv / (1.0f + expf(-gv)) * uv;
                if (!(fabsf(h) <= 65504.0f)) record_status(a.status, MOE_ERR_UNSUPPORTED);
                H[static_cast<size_t>(m.row0 + c0 + c) * Icur + n] = __half_as_ushort(__float2half_rn(h));
              }
            }
          }
        }
      } else {
        // destination slot and routing weight of each column, loaded once per
        // item: lane L owns columns L, L+32, L+64, L+96
        int slot[4];
        float wt[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = lane + 32 * i;
          slot[i] = -1;
          wt[i] = 0.0f;
          if (c < m.rows) {
            const int p = m.row0 + c;
            if (m.shared) {
              slot[i] = p * (a.k + 1) + a.k;
              wt[i] = 1.0f;
            } else {
              const int asg = __ldg(a.perm + p);
              if (asg >= 0 && asg < a.T * a.k) {
                slot[i] = asg + asg / a.k;
                wt[i] = __ldg(a.w + asg);
              } else {
                record_status(a.status, MOE_ERR_INVALID_ARG);
              }
            }
          }
        }
        for (int c0 = 0; c0 < bn; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tbase + c0, v);
          tc_wait_ld();
          const int grp = c0 >> 5;  // which register holds these columns (uniform in the warp)
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int col = c0 + c;
            const int src = col & 31;
            int sl;
            float wv;
            if (grp == 0) {
              sl = __shfl_sync(0xffffffffu, slot[0], src);
              wv = __shfl_sync(0xffffffffu, wt[0], src);
            } else if (grp == 1) {
              sl = __shfl_sync(0xffffffffu, slot[1], src);
              wv = __shfl_sync(0xffffffffu, wt[1], src);
            } else if (grp == 2) {
              sl = __shfl_sync(0xffffffffu, slot[2], src);
              wv = __shfl_sync(0xffffffffu, wt[2], src);
            } else {
              sl = __shfl_sync(0xffffffffu, slot[3], src);
              wv = __shfl_sync(0xffffffffu, wt[3], src);
            }
            if (n < a.d && sl >= 0) a.ypart[static_cast<size_t>(sl) * a.d + n] = wv * __uint_as_float(v[c]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
      if (kGateUp) {
        accphase ^= 1;
      } else if (++accb == 2) {
        accb = 0;
        accphase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// X (bf16) -> fp16 copy used as the tensor-core operand.  Values outside the
// fp16 range are recorded as MOE_ERR_UNSUPPORTED.
__global__ void x_to_f16_kernel(const uint16_t* __restrict__ X, size_t n8, uint16_t* __restrict__ Xh,
                                uint32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  bool range_ok = true;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(X)[i];
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(in[j] << 16);
      const float hi = __uint_as_float(in[j] & 0xFFFF0000u);
      range_ok &= fabsf(lo) <= 65504.0f && fabsf(hi) <= 65504.0f;
      out[j] = f32x2_to_f16x2(lo, hi);
    }
    reinterpret_cast<uint4*>(Xh)[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
  if (!range_ok) record_status(status, MOE_ERR_UNSUPPORTED);
}

// Y[t] = bf16( sum over the k routed slots and the shared slot )
__global__ void combine_kernel(const float* __restrict__ ypart, int T, int d, int stride_slots, int slots,
                               uint16_t* __restrict__ Y) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t total4 = static_cast<size_t>(T) * d / 4;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t e = i * 4;
    const size_t t = e / d;
    const size_t n = e % d;
    const float4* src = reinterpret_cast<const float4*>(ypart + t * stride_slots * d + n);
    float4 acc = src[0];
    for (int j = 1; j < slots; ++j) {
      const float4 v = src[static_cast<size_t>(j) * d / 4];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.x))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.y))) << 16);
    const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.z))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.w))) << 16);
    *reinterpret_cast<uint2*>(Y + e) = make_uint2(lo, hi);
  }
}

bool g_gemm_attr = false;

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, const GemmMaps* routed, const GemmMaps* shared, const GemmActMaps* act,
                        cudaStream_t stream, bool pdl) {
  using CG = Cfg<true>;
  using CD = Cfg<false>;
  if (!g_gemm_attr) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CG::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(moe_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, CD::kSmemBytes);
    if (e != cudaSuccess) return e;
    g_gemm_attr = true;
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
  cfg.blockDim = dim3(kThreads);

  {
    cudaLaunchConfig_t c2 = cfg;
    c2.gridDim = dim3(a.num_sms * 2);
    c2.blockDim = dim3(256);
    c2.dynamicSmemBytes = 0;
    const size_t n8 = static_cast<size_t>(a.T) * a.d / 8;
    timer_begin(kKToF16, stream);
    cudaError_t e = cudaLaunchKernelEx(&c2, x_to_f16_kernel, a.X, n8, a.Xh, a.status);
    timer_end(kKToF16, stream);
    if (e != cudaSuccess) return e;
  }
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.dynamicSmemBytes = CG::kSmemBytes;
  timer_begin(kKGemmGateUp, stream);
  cudaError_t err = cudaLaunchKernelEx(&cfg, moe_gemm_kernel<true>, routed->q_gate, routed->q_up, routed->sb_gate,
                                       routed->sb_up, sh->q_gate, sh->q_up, sh->sb_gate, sh->sb_up, act->x, act->x, a);
  timer_end(kKGemmGateUp, stream);
  if (err != cudaSuccess) return err;

  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.dynamicSmemBytes = CD::kSmemBytes;
  timer_begin(kKGemmDown, stream);
  err = cudaLaunchKernelEx(&cfg, moe_gemm_kernel<false>, routed->q_down, routed->q_down, routed->sb_down,
                           routed->sb_down, sh->q_down, sh->q_down, sh->sb_down, sh->sb_down, act->h_routed,
                           act->h_shared, a);
  timer_end(kKGemmDown, stream);
  if (err != cudaSuccess) return err;

  cfg.gridDim = dim3(a.num_sms * 4);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  const int slots = a.k + (a.I_shared > 0 ? 1 : 0);
  timer_begin(kKCombine, stream);
  err = cudaLaunchKernelEx(&cfg, combine_kernel, static_cast<const float*>(a.ypart), a.T, a.d, a.k + 1, slots, a.Y);
  timer_end(kKCombine, stream);
  return err;
}

}  // namespace bm
