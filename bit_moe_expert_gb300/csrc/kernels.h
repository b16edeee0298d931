// Launch entry points of the kernels, called by the host boundary (api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "status.h"

namespace bm {

// Kernel kinds for the optional per-kernel timing (moe_profile.h).
enum KernelKind {
  kKRoute = 0,
  kKDecode,    // the fused decode kernel (gate/up + down)
  kKRouter,    // the router projection
  kKXGather,
  kKGemmGateUp,
  kKGemmDown,
  kKCombine,
  kKPrepack,
  kKTopkWide,  // exact top-K of wide rows
  kKernelKinds
};
void timer_begin(int id, cudaStream_t s);
void timer_end(int id, cudaStream_t s);

struct RouteOut {
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* block_map;
  int32_t* num_blocks;
};

// One-time launch set-up, per device and kernel, thread-safe: raise the
// kernel's dynamic shared-memory limit to at least `bytes`; the kernel's
// resident CTAs per SM at (threads, smem).
cudaError_t set_max_dynamic_smem(const void* func, int bytes);
cudaError_t occupancy_per_sm(const void* func, int threads, size_t smem, int* per_sm);

size_t route_hist_elems(int T, int E);
// status: where device-side errors go (null: the workspace header's status word)
cudaError_t launch_route(const float* logits, int T, int E, int k, int block_rows, const RouteOut& out, void* ws,
                         cudaStream_t stream, bool pdl, uint32_t* status = nullptr);
cudaError_t launch_prepack_codes(const uint32_t* q, int E, int N, int K, int bits, uint32_t* qp,
                                 cudaStream_t stream);
cudaError_t launch_prepack(const uint16_t* scale, const uint16_t* bias, int E, int N, int K, uint32_t* sb,
                           cudaStream_t stream);
// fp16 weights W [E][N][K] = q * scale + bias of one prepacked matrix (bits per code 2, 3 or 4)
cudaError_t launch_dequant(const uint32_t* qp, const uint32_t* sb, int E, int N, int K, int bits, uint16_t* W,
                           cudaStream_t stream);

// Router projection: logits [T][E] fp32 = X [T][d] bf16 times Wr [E][d] bf16
// transposed (d a multiple of 32).  With `maps` (router_tc_shape true), the
// tensor-core path: TMA tiles, tcgen05 MMAs, K split over a 4-CTA cluster.
constexpr int kRouterTcE = 128;     // experts per CTA (the MMA's M)
constexpr int kRouterTcT = 64;      // tokens per CTA (the MMA's N)
constexpr int kRouterTcSplit = 4;   // CTAs of a cluster, each a quarter of K
struct RouterMaps {
  CUtensorMap x;   // X [T][d] bf16, box (64, kRouterTcT), 128-byte swizzle
  CUtensorMap wr;  // Wr [E][d] bf16, box (64, kRouterTcE), 128-byte swizzle
};
bool router_tc_shape(int T, int d, int E);
cudaError_t launch_router(const uint16_t* X, int T, int d, const uint16_t* Wr, int E, float* logits,
                          const RouterMaps* maps, cudaStream_t stream, bool pdl);

// Exact top-K (K <= 64) of each row of logits [T][V] (V <= 2^20): values and
// indices [T][K], descending, a lower index first among equal values.
size_t topk_wide_smem_bytes(int V, int K);
cudaError_t launch_topk_wide(const float* logits, int T, int V, int K, float* values, int32_t* indices,
                             int num_sms, cudaStream_t stream, bool pdl);

// ---------------------------------------------------------------- decode GEMV
constexpr int kDecodeRowsGU = 32;      // gate/up rows per item (phase 1)
constexpr int kDecodeChunkGroups = 8;  // 64-column groups per gate/up stage
constexpr int kDecodeRowsDown = 16;    // output rows per block (phase 2)

// Tensor maps of one expert set for the decode kernel.
struct DecodeMaps {
  CUtensorMap q_gate, q_up;    // codes [E][d/64][I*wpg], box (32 rows * wpg words, kDecodeChunkGroups groups, 1)
  CUtensorMap sb_gate, sb_up;  // group parameters [E][d/64][I], box (32 rows, d/64 groups, 1)
  CUtensorMap q_down;          // codes [E][I/64][d*wpg], box (16 rows * wpg words, I/64 groups, 1)
  CUtensorMap sb_down;         // group parameters [E][I/64][d], box (16 rows, I/64 groups, 1)
};

struct DecodeArgs {
  const uint16_t* X;      // [T][d] bf16
  const int32_t* ids;     // [T][k] (routing read from memory)
  const float* w;         // [T][k]
  const float* logits;    // [T][E]: when not null the kernel routes its own tokens (E <= 256) and its last
                          // CTA writes every routing output to `out`
  RouteOut out;           // routing outputs written by the kernel (logits != null)
  int block_rows;         // tile height of the block map it writes
  uint16_t* Y;            // [T][d] bf16
  uint8_t* hbuf;          // h records of the call's slots, decode_scratch_bytes, 16-byte aligned
  // gate and up codes of the routed experts and of the shared expert (the prepacked [E][d/64][I][wpg] arrays),
  // read directly into registers when every CTA has at most one phase-1 item
  const uint32_t *qg_r, *qu_r, *qg_s, *qu_s;
  uint32_t* status;
  int T, d, I, k, I_shared, E, num_sms;
  int bits;  // bits per weight code: 4 or 2
};

bool decode_supported(int T, int d, int I, int I_shared, int k);
size_t decode_scratch_bytes(int T, int I, int I_shared);  // global scratch: the h records
cudaError_t launch_decode(const DecodeArgs& a, const DecodeMaps* routed, const DecodeMaps* shared, void* ws,
                          cudaStream_t stream, bool pdl);
// Test hooks of the decode kernel: the limit of the wait at its barrier over
// the grid in SM clock cycles (<= 0: the default of about 2 s), and one CTA
// (-1: none) whose arrival at that barrier is skipped, so that the wait runs
// out.
cudaError_t decode_debug(long long wait_limit_cycles, int drop_cta);

// ---------------------------------------------------------------- prefill GEMM
constexpr int kGemmBM = 128;   // weight rows per tile (MMA M)
constexpr int kGemmBK = 64;    // K of one quantisation group
constexpr int kGemmGroupsGU = 2;    // quantisation groups per pipeline stage, gate/up GEMM
constexpr int kGemmGroupsDown = 2;  // ... down GEMM
constexpr int kGemmBN = 128;   // max tokens per tile (MMA N)

struct GemmMaps {
  // codes, box (wpg words, 128 rows, groups per stage); 32-byte swizzle for 4-bit codes.  3-bit codes: box
  // (64 rows x 3 units, 1)
  CUtensorMap q_gate, q_up, q_down;
  CUtensorMap sb_gate, sb_up, sb_down;  // group parameters, box (128 rows, groups per stage, 1)
};

struct GemmArgs {
  const int32_t* perm;        // [A]
  const int32_t* inv_perm;    // [A]
  const int32_t* block_map;   // [nb][3]
  const int32_t* num_blocks;  // [1]
  const float* w;             // [A]
  float* ypart;               // [A + T][d] fp32 expert outputs: routed rows in permuted order, then shared rows
  uint16_t* h_routed;         // [A][I] fp16
  uint16_t* h_shared;         // [T][I_shared] fp16
  const uint16_t* X;          // [T][d] bf16 input
  uint16_t* Xh;               // [A + T][d] fp16 gathered rows of X (tensor-core operand)
  uint16_t* Y;                // [T][d] bf16
  uint32_t* status;
  int T, d, I, k, I_shared, E, num_sms, max_blocks;
  int bits;  // bits per weight code: 4, 3 or 2
};

struct GemmActMaps {
  CUtensorMap x;         // gathered X [A + T][d] fp16, box (64, kGemmBN), 128-byte swizzle
  CUtensorMap h_routed;  // H [A][I] fp16, box (64, kGemmBN), 128-byte swizzle
  CUtensorMap h_shared;  // H [T][I_shared] fp16, same box
  CUtensorMap ypart;     // expert outputs [A + T][d] fp32, box (32, 16): the down GEMM's stores
};

cudaError_t launch_gemm(const GemmArgs& a, const GemmMaps* routed, const GemmMaps* shared, const GemmActMaps* act,
                        cudaStream_t stream, bool pdl);

}  // namespace bm
