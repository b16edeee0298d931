// Host side of the C ABI declared in include/moe.h: argument validation,
// workspace layout, TMA tensor-map encoding and kernel launches.  Nothing here
// allocates device memory or synchronises, except moe_check_status.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "moe.h"

namespace bm {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Encoded tensor maps, reused across calls: a map is a pure function of its
// arguments, and a layer call encodes a dozen of them (about a microsecond of
// host time each), which is most of the host cost of a decode-layer call.  A
// direct-mapped table keyed by every argument; a hit copies the stored map.
struct MapKey {
  const void* ptr;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3];
  int rank, dt, sw;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kMapCache = 256;
MapEntry g_maps[kMapCache];
std::mutex g_maps_mu;

bool encode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* ptr, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));  // padding bytes take part in the comparison
  const bool cacheable = rank >= 1 && rank <= 3;
  if (cacheable) {
    key.ptr = ptr;
    for (int i = 0; i < rank; ++i) {
      key.dims[i] = dims[i];
      key.box[i] = box[i];
      if (i + 1 < rank) key.strides[i] = strides[i];
    }
    key.rank = rank;
    key.dt = static_cast<int>(dt);
    key.sw = static_cast<int>(sw);
    uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's bytes
    const unsigned char* kb = reinterpret_cast<const unsigned char*>(&key);
    for (size_t i = 0; i < sizeof(key); ++i) h = (h ^ kb[i]) * 1099511628211ull;
    const int slot = static_cast<int>(h % kMapCache);
    {
      std::lock_guard<std::mutex> lock(g_maps_mu);
      if (g_maps[slot].used && g_maps[slot].key == key) {
        *map = g_maps[slot].map;
        return true;
      }
    }
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = g_encode(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lock(g_maps_mu);
    std::memcpy(&g_maps[slot].key, &key, sizeof(key));  // keys compare as bytes
    g_maps[slot].map = *map;
    g_maps[slot].used = true;
    return true;
  }
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// codes q [E][K/64][N][wpg] uint32 (group-major, moe_prepack_codes; wpg = 2 x
// bits per code words per row and group), seen as a 3-D tensor
// [E*K/64][N][wpg]; a box covers box_rows rows of box_groups consecutive groups
bool encode_codes(CUtensorMap* map, const uint32_t* q, int E, int N, int K, cuuint32_t box_rows,
                  cuuint32_t box_groups, CUtensorMapSwizzle sw, int wpg) {
  const int G = K / 64;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(wpg), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(E) * G};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(wpg) * 4, static_cast<cuuint64_t>(N) * wpg * 4};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(wpg), box_rows, box_groups};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, q, dims, strides, box, sw);
}

// The same codes seen as [E][K/64][N*wpg]: the pieces of consecutive rows of
// one group are contiguous, so a box of box_rows rows (box_rows*wpg*4 bytes,
// at most 1 KiB) is one line; box_groups consecutive groups of one expert
// (groups past the last read as zeros)
bool encode_codes_rows(CUtensorMap* map, const uint32_t* q, int E, int N, int K, cuuint32_t box_rows,
                       cuuint32_t box_groups, int wpg) {
  const int G = K / 64;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N) * wpg, static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * wpg * 4, static_cast<cuuint64_t>(N) * wpg * 4 * G};
  const cuuint32_t box[3] = {box_rows * static_cast<cuuint32_t>(wpg), box_groups, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 3-bit codes q [E][K/64][N][6] uint32 seen as [E*K/64][N*3] 8-byte units:
// a row's 24 bytes are three units, so a box of box_rows rows (box_rows*3
// units, at most 256) starts on a 16-byte boundary whenever its first row is
// even; rows past N read as zeros
bool encode_codes3(CUtensorMap* map, const uint32_t* q, int E, int N, int K, cuuint32_t box_rows) {
  const int G = K / 64;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N) * 3, static_cast<cuuint64_t>(E) * G};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 24};
  const cuuint32_t box[2] = {box_rows * 3, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// fp16 activations [rows][cols]: boxes of 64 columns (128 bytes) x kGemmBN
// rows, 128-byte swizzle (the K-major operand layout of the tensor cores)
bool encode_act(CUtensorMap* map, const uint16_t* p, int rows, int cols) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kGemmBN)};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// fp32 expert outputs [rows][cols]: boxes of 32 columns x 16 rows (the down
// GEMM's epilogue stores one warp's 32 weight rows for 16 tokens at a time)
bool encode_out(CUtensorMap* map, const float* p, int rows, int cols) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  const cuuint32_t box[2] = {32, 16};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// bf16 rows [rows][cols] (the router projection's X and W_r): boxes of 64
// columns (128 bytes) x box_rows rows, 128-byte swizzle; rows past the end
// read as zeros
bool encode_bf16_rows(CUtensorMap* map, const uint16_t* p, int rows, int cols, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// group parameters sb [E][K/64][N] uint32
bool encode_groups(CUtensorMap* map, const uint32_t* sb, int E, int N, int K, cuuint32_t box_rows,
                   cuuint32_t box_groups) {
  const int G = K / 64;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 4, static_cast<cuuint64_t>(N) * 4 * G};
  const cuuint32_t box[3] = {box_rows, box_groups, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, sb, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int g_sm_count[64] = {0};

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

bool env_flag(const char* name, bool dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return !(v[0] == '0' || v[0] == 'n' || v[0] == 'N' || v[0] == 'f' || v[0] == 'F');
}

enum class Path { kGemv, kGemm };

// Forward workspace: header, then one region used by either path.
struct FwdLayout {
  size_t dec_h;                                              // h records of the decode kernel
  size_t gemm_h_routed, gemm_h_shared, gemm_ypart, gemm_xh;  // fp16, fp16, fp32, fp16
  size_t total;
};

FwdLayout fwd_layout(int T, int d, int I, int k, int I_shared) {
  FwdLayout L;
  const size_t A = static_cast<size_t>(T) * k;
  size_t o = sizeof(WsHeader);
  const size_t base = o;
  L.dec_h = o;
  o = round256(o + (T <= kGemvMaxT ? decode_scratch_bytes(T, I, I_shared) : 0));
  const size_t dec_end = o;
  o = base;
  L.gemm_h_routed = o;
  o = round256(o + A * I * 2);
  L.gemm_h_shared = o;
  o = round256(o + static_cast<size_t>(T) * I_shared * 2);
  L.gemm_ypart = o;
  o = round256(o + (A + static_cast<size_t>(T)) * d * 4);
  L.gemm_xh = o;
  o = round256(o + (A + static_cast<size_t>(T)) * d * 2);
  L.total = o > dec_end ? o : dec_end;
  return L;
}

bool qmat_ok(const moe_qmat& m) { return m.q && m.sb && aligned16(m.q) && aligned16(m.sb); }

bool experts_ok(const moe_experts* ex) {
  return ex && qmat_ok(ex->gate) && qmat_ok(ex->up) && qmat_ok(ex->down) && ex->n_experts >= 1 &&
         (ex->bits == 0 || (ex->bits >= 2 && ex->bits <= 4));
}

int code_bits(const moe_experts* ex) { return ex->bits == 0 ? 4 : ex->bits; }

// One-time launch set-up shared by the launchers: the dynamic shared-memory
// limit of a kernel and its resident CTAs per SM, per device (both depend on
// the device's context), under one lock, since host threads may make their
// first calls on different devices at the same time.
struct FuncEntry {
  int dev;
  const void* func;
  int threads;
  size_t smem;
  int value;  // the limit set (attribute entries, threads = -1), or CTAs per SM
};
constexpr int kFuncEntries = 128;
FuncEntry g_func[kFuncEntries];
int g_func_n = 0;
std::mutex g_func_mu;

}  // namespace

cudaError_t set_max_dynamic_smem(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_func_mu);
  for (int i = 0; i < g_func_n; ++i)
    if (g_func[i].dev == dev && g_func[i].func == func && g_func[i].threads == -1) {
      if (g_func[i].value >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) g_func[i].value = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && g_func_n < kFuncEntries) g_func[g_func_n++] = FuncEntry{dev, func, -1, 0, bytes};
  return e;
}

cudaError_t occupancy_per_sm(const void* func, int threads, size_t smem, int* per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_func_mu);
  for (int i = 0; i < g_func_n; ++i)
    if (g_func[i].dev == dev && g_func[i].func == func && g_func[i].threads == threads && g_func[i].smem == smem) {
      *per_sm = g_func[i].value;
      return cudaSuccess;
    }
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem);
  if (e != cudaSuccess) return e;
  if (g_func_n < kFuncEntries) g_func[g_func_n++] = FuncEntry{dev, func, threads, smem, n};
  *per_sm = n;
  return cudaSuccess;
}

}  // namespace bm

using namespace bm;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE";
  }
  return "MOE_ERR_UNKNOWN";
}

int moe_device_sm_count(void) { return sm_count(); }

size_t moe_prepack_bytes(int E, int N, int K) {
  if (E < 1 || N < 1 || K < 64 || K % 64) return 0;
  return static_cast<size_t>(E) * (K / 64) * N * 4;
}

moe_status moe_prepack_codes_bits(const uint32_t* q, int E, int N, int K, int bits, uint32_t* qp,
                                  moe_stream stream) {
  if (!q || !qp || E < 1 || N < 1 || K < 64 || K % 64 != 0 || !aligned16(q) || !aligned16(qp))
    return MOE_ERR_INVALID_ARG;
  if (bits < 2 || bits > 4) return MOE_ERR_INVALID_ARG;
  if (launch_prepack_codes(q, E, N, K, bits, qp, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_prepack_codes(const uint32_t* q, int E, int N, int K, uint32_t* qp, moe_stream stream) {
  return moe_prepack_codes_bits(q, E, N, K, 4, qp, stream);
}

moe_status moe_prepack_scales(const uint16_t* scale, const uint16_t* bias, int E, int N, int K, uint32_t* sb,
                              moe_stream stream) {
  if (!scale || !bias || !sb || E < 1 || N < 1 || K < 64 || K % 64) return MOE_ERR_INVALID_ARG;
  if (launch_prepack(scale, bias, E, N, K, sb, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_dequant_experts(const moe_qmat* m, int E, int N, int K, int bits, uint16_t* W, moe_stream stream) {
  if (!m || !W || E < 1 || N < 1 || K < 64 || K % 64) return MOE_ERR_INVALID_ARG;
  if (bits < 2 || bits > 4) return MOE_ERR_INVALID_ARG;
  if (!qmat_ok(*m) || !aligned16(W)) return MOE_ERR_INVALID_ARG;
  if (launch_dequant(m->q, m->sb, E, N, K, bits, W, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_route_max_blocks(int T, int E, int k, int block_rows) {
  if (T < 0 || E < 1 || k < 1 || block_rows < 1) return 0;
  const long long A = static_cast<long long>(T) * k;
  return static_cast<int>((A + block_rows - 1) / block_rows + E);
}

size_t moe_route_workspace_bytes(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  const size_t A = static_cast<size_t>(T) * k;
  return round256(sizeof(WsHeader) + (route_hist_elems(T, E) + A) * 4);
}

moe_status moe_route(const float* logits, int T, int E, int k, int block_rows, moe_routing* out, void* ws,
                     size_t ws_bytes, moe_stream stream) {
  if (!out || T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > kMaxK || k > E) return MOE_ERR_UNSUPPORTED;
  if (block_rows < 1 || block_rows > kMaxBlockRows) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * k > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  // arrays of length T*k may be null when T = 0
  if (!out->counts || !out->offsets || !out->block_map || !out->num_blocks) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !out->ids || !out->w || !out->perm || !out->inv_perm)) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < moe_route_workspace_bytes(T, E, k))
    return MOE_ERR_WORKSPACE;
  out->block_rows = block_rows;
  RouteOut o{out->ids, out->w, out->counts, out->offsets, out->perm, out->inv_perm, out->block_map, out->num_blocks};
  const bool pdl = env_flag("MOE_PDL", true);
  if (launch_route(logits, T, E, k, block_rows, o, ws, reinterpret_cast<cudaStream_t>(stream), pdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_router_logits(const uint16_t* X, int T, int d, const uint16_t* W_r, int E, float* logits,
                             moe_stream stream) {
  if (T < 0 || d < 64 || d % 64 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!X || !W_r || !logits)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W_r)) & 15u)) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * E > (1ll << 31) - 1) return MOE_ERR_UNSUPPORTED;
  const bool pdl = env_flag("MOE_PDL", true);
  // the tensor-core shape wants 16-byte rows of logits for its vector stores;
  // MOE_ROUTER_TC=0 keeps the warp-MMA shapes (for comparisons)
  RouterMaps maps;
  const RouterMaps* mp = nullptr;
  if (router_tc_shape(T, d, E) && !(reinterpret_cast<uintptr_t>(logits) & 15u) && env_flag("MOE_ROUTER_TC", true)) {
    if (!get_encoder() || !encode_bf16_rows(&maps.x, X, T, d, kRouterTcT) ||
        !encode_bf16_rows(&maps.wr, W_r, E, d, kRouterTcE))
      return MOE_ERR_CUDA;
    mp = &maps;
  }
  if (launch_router(X, T, d, W_r, E, logits, mp, reinterpret_cast<cudaStream_t>(stream), pdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_route_x(const uint16_t* X, int T, int d, const uint16_t* W_r, int E, int k, int block_rows,
                       float* logits, moe_routing* out, void* ws, size_t ws_bytes, moe_stream stream) {
  // every argument moe_route checks, before anything is launched
  if (!out || T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > kMaxK || k > E) return MOE_ERR_UNSUPPORTED;
  if (block_rows < 1 || block_rows > kMaxBlockRows) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * k > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  if (!out->counts || !out->offsets || !out->block_map || !out->num_blocks) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!out->ids || !out->w || !out->perm || !out->inv_perm)) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < moe_route_workspace_bytes(T, E, k))
    return MOE_ERR_WORKSPACE;
  const moe_status st = moe_router_logits(X, T, d, W_r, E, logits, stream);
  if (st != MOE_OK) return st;
  return moe_route(logits, T, E, k, block_rows, out, ws, ws_bytes, stream);
}

moe_status moe_topk_wide(const float* logits, int T, int V, int K, float* values, int32_t* indices,
                         moe_stream stream) {
  if (T < 0 || K < 1 || V < K) return MOE_ERR_INVALID_ARG;
  if (K > 64 || V > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!logits || !values || !indices)) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) & 3u) return MOE_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  const bool pdl = env_flag("MOE_PDL", true);
  if (launch_topk_wide(logits, T, V, K, values, indices, sms, reinterpret_cast<cudaStream_t>(stream), pdl) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

size_t moe_forward_workspace_bytes(int T, int d, int I, int E, int k, int I_shared) {
  if (T < 0 || d < 1 || I < 1 || E < 1 || k < 1 || I_shared < 0) return 0;
  return fwd_layout(T, d, I, k, I_shared).total;
}

namespace {

// moe_forward; with `logits` set and T on the decode path, the decode kernel
// also routes the tokens and writes every routing output to *r (moe_layer).
// The decode kernel's twelve tensor maps for one (routed, shared) expert set
// and shape, built once and reused: a decode-layer call then spends no host
// time on encoding.  Keyed by every pointer and size the maps depend on.
struct DecodeMapsKey {
  const void* p[12];
  int E, d, I, I_shared, wpg;
  bool operator==(const DecodeMapsKey& o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};
struct DecodeMapsEntry {
  DecodeMapsKey key;
  DecodeMaps mr, ms;
  bool used;
};
constexpr int kDecodeMapsCache = 64;
DecodeMapsEntry g_dmaps[kDecodeMapsCache];
std::mutex g_dmaps_mu;

bool decode_maps(const moe_experts* routed, const moe_experts* shared, int E, int d, int I, int I_shared, int wpg,
                 DecodeMaps* mr, DecodeMaps* ms) {
  DecodeMapsKey key;
  std::memset(&key, 0, sizeof(key));
  const moe_qmat* mats[6] = {&routed->gate, &routed->up, &routed->down, shared ? &shared->gate : nullptr,
                             shared ? &shared->up : nullptr, shared ? &shared->down : nullptr};
  for (int i = 0; i < 6; ++i) {
    key.p[2 * i] = mats[i] ? mats[i]->q : nullptr;
    key.p[2 * i + 1] = mats[i] ? mats[i]->sb : nullptr;
  }
  key.E = E;
  key.d = d;
  key.I = I;
  key.I_shared = shared ? I_shared : 0;
  key.wpg = wpg;
  uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's bytes
  const unsigned char* kb = reinterpret_cast<const unsigned char*>(&key);
  for (size_t i = 0; i < sizeof(key); ++i) h = (h ^ kb[i]) * 1099511628211ull;
  DecodeMapsEntry& slot = g_dmaps[h % kDecodeMapsCache];
  {
    std::lock_guard<std::mutex> lock(g_dmaps_mu);
    if (slot.used && slot.key == key) {
      *mr = slot.mr;
      *ms = slot.ms;
      return true;
    }
  }
  const cuuint32_t G1 = static_cast<cuuint32_t>(d / 64), G2 = static_cast<cuuint32_t>(I / 64);
  bool ok = encode_codes_rows(&mr->q_gate, routed->gate.q, E, I, d, kDecodeRowsGU, kDecodeChunkGroups, wpg) &&
            encode_codes_rows(&mr->q_up, routed->up.q, E, I, d, kDecodeRowsGU, kDecodeChunkGroups, wpg) &&
            encode_codes_rows(&mr->q_down, routed->down.q, E, d, I, kDecodeRowsDown, G2, wpg) &&
            encode_groups(&mr->sb_gate, routed->gate.sb, E, I, d, kDecodeRowsGU, G1) &&
            encode_groups(&mr->sb_up, routed->up.sb, E, I, d, kDecodeRowsGU, G1) &&
            encode_groups(&mr->sb_down, routed->down.sb, E, d, I, kDecodeRowsDown, G2);
  if (ok && shared) {
    const cuuint32_t G2s = static_cast<cuuint32_t>(I_shared / 64);
    ok = encode_codes_rows(&ms->q_gate, shared->gate.q, 1, I_shared, d, kDecodeRowsGU, kDecodeChunkGroups, wpg) &&
         encode_codes_rows(&ms->q_up, shared->up.q, 1, I_shared, d, kDecodeRowsGU, kDecodeChunkGroups, wpg) &&
         encode_codes_rows(&ms->q_down, shared->down.q, 1, d, I_shared, kDecodeRowsDown, G2s, wpg) &&
         encode_groups(&ms->sb_gate, shared->gate.sb, 1, I_shared, d, kDecodeRowsGU, G1) &&
         encode_groups(&ms->sb_up, shared->up.sb, 1, I_shared, d, kDecodeRowsGU, G1) &&
         encode_groups(&ms->sb_down, shared->down.sb, 1, d, I_shared, kDecodeRowsDown, G2s);
  }
  if (!ok) return false;
  std::lock_guard<std::mutex> lock(g_dmaps_mu);
  std::memcpy(&slot.key, &key, sizeof(key));  // padding included: keys compare as bytes
  slot.mr = *mr;
  slot.ms = *ms;
  slot.used = true;
  return true;
}

moe_status forward_impl(const uint16_t* X, int T, int d, int I, int k, const moe_experts* routed,
                        const moe_experts* shared, int I_shared, const moe_routing* r, uint16_t* Y, void* ws,
                        size_t ws_bytes, moe_stream stream, const float* logits) {
  if (T < 0 || d < 64 || I < 64 || k < 1 || I_shared < 0) return MOE_ERR_INVALID_ARG;
  if (d % 64 || I % 64 || I_shared % 64) return MOE_ERR_INVALID_ARG;
  if ((shared != nullptr) != (I_shared > 0)) return MOE_ERR_INVALID_ARG;
  if (!experts_ok(routed) || (shared && (!experts_ok(shared) || shared->n_experts != 1)))
    return MOE_ERR_INVALID_ARG;
  const int bits = code_bits(routed);
  if (shared && code_bits(shared) != bits) return MOE_ERR_INVALID_ARG;
  const int wpg = 2 * bits;  // code words per row and group
  const int E = routed->n_experts;
  if (E > kMaxE || k > kMaxK || k > E) return MOE_ERR_UNSUPPORTED;
  if (!r) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
      ws_bytes < moe_forward_workspace_bytes(T, d, I, E, k, I_shared))
    return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  if (!r->ids || !r->w || !r->perm || !r->block_map || !r->num_blocks) return MOE_ERR_INVALID_ARG;
  if (!X || !Y || !aligned16(X) || !aligned16(Y)) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * k > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  if (!get_encoder()) return MOE_ERR_CUDA;

  const FwdLayout L = fwd_layout(T, d, I, k, I_shared);
  char* wsb = static_cast<char*>(ws);
  uint32_t* status = &static_cast<WsHeader*>(ws)->status;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool pdl = env_flag("MOE_PDL", true);

  // Path: decode kernels for small T unless their shared-memory plan does not fit.
  Path path = T <= kGemvMaxT ? Path::kGemv : Path::kGemm;
  if (const char* p = std::getenv("MOE_PATH")) {
    if (!std::strcmp(p, "gemv")) path = Path::kGemv;
    if (!std::strcmp(p, "gemm")) path = Path::kGemm;
  }
  if (path == Path::kGemv && !decode_supported(T, d, I, I_shared, k)) {
    if (T > kGemvMaxT) return MOE_ERR_UNSUPPORTED;  // the decode kernel takes at most kGemvMaxT tokens
    path = Path::kGemm;
  }

  if (path == Path::kGemv) {
    DecodeMaps mr, ms;
    if (!decode_maps(routed, shared, E, d, I, I_shared, wpg, &mr, &ms)) return MOE_ERR_CUDA;
    DecodeArgs a{};
    a.X = X;
    a.ids = r->ids;
    a.w = r->w;
    a.logits = logits;
    a.out = RouteOut{r->ids, r->w, r->counts, r->offsets, r->perm, r->inv_perm, r->block_map, r->num_blocks};
    a.block_rows = r->block_rows;
    a.Y = Y;
    a.hbuf = reinterpret_cast<uint8_t*>(wsb + L.dec_h);
    a.qg_r = routed->gate.q;
    a.qu_r = routed->up.q;
    a.qg_s = shared ? shared->gate.q : nullptr;
    a.qu_s = shared ? shared->up.q : nullptr;
    a.status = status;
    a.T = T;
    a.d = d;
    a.I = I;
    a.k = k;
    a.I_shared = I_shared;
    a.E = E;
    a.num_sms = sm_count();
    a.bits = bits;
    if (a.num_sms <= 0) return MOE_ERR_CUDA;
    if (launch_decode(a, &mr, shared ? &ms : nullptr, ws, st, pdl) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }

  if (r->block_rows < 1 || r->block_rows > kGemmBN) return MOE_ERR_UNSUPPORTED;
  const int A = T * k;
  // a row's codes of one group: 32 bytes (4-bit) read through a 32-byte
  // swizzle, or 16 bytes (2-bit), already conflict-free; 24 bytes (3-bit) in
  // two boxes of 64 rows, read as 8-byte units (conflict-free too)
  const CUtensorMapSwizzle code_swizzle = bits == 4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE;
  auto enc_q = [&](CUtensorMap* map, const uint32_t* q, int ne, int N, int K, int groups) {
    return bits == 3 ? encode_codes3(map, q, ne, N, K, kGemmBM / 2)
                     : encode_codes(map, q, ne, N, K, kGemmBM, groups, code_swizzle, wpg);
  };
  GemmMaps mr, ms;
  GemmActMaps act;
  uint16_t* hr = reinterpret_cast<uint16_t*>(wsb + L.gemm_h_routed);
  uint16_t* hs = reinterpret_cast<uint16_t*>(wsb + L.gemm_h_shared);
  uint16_t* xh = reinterpret_cast<uint16_t*>(wsb + L.gemm_xh);
  bool ok = enc_q(&mr.q_gate, routed->gate.q, E, I, d, kGemmGroupsGU) &&
            enc_q(&mr.q_up, routed->up.q, E, I, d, kGemmGroupsGU) &&
            enc_q(&mr.q_down, routed->down.q, E, d, I, kGemmGroupsDown) &&
            encode_groups(&mr.sb_gate, routed->gate.sb, E, I, d, kGemmBM, kGemmGroupsGU) &&
            encode_groups(&mr.sb_up, routed->up.sb, E, I, d, kGemmBM, kGemmGroupsGU) &&
            encode_groups(&mr.sb_down, routed->down.sb, E, d, I, kGemmBM, kGemmGroupsDown) &&
            encode_act(&act.x, xh, A + (shared ? T : 0), d) && encode_act(&act.h_routed, hr, A, I) &&
            encode_out(&act.ypart, reinterpret_cast<const float*>(wsb + L.gemm_ypart), A + (shared ? T : 0), d);
  if (ok && shared)
    ok = enc_q(&ms.q_gate, shared->gate.q, 1, I_shared, d, kGemmGroupsGU) &&
         enc_q(&ms.q_up, shared->up.q, 1, I_shared, d, kGemmGroupsGU) &&
         enc_q(&ms.q_down, shared->down.q, 1, d, I_shared, kGemmGroupsDown) &&
         encode_groups(&ms.sb_gate, shared->gate.sb, 1, I_shared, d, kGemmBM, kGemmGroupsGU) &&
         encode_groups(&ms.sb_up, shared->up.sb, 1, I_shared, d, kGemmBM, kGemmGroupsGU) &&
         encode_groups(&ms.sb_down, shared->down.sb, 1, d, I_shared, kGemmBM, kGemmGroupsDown) &&
         encode_act(&act.h_shared, hs, T, I_shared);
  if (ok && !shared) act.h_shared = act.h_routed;  // never read without a shared expert
  if (!ok) return MOE_ERR_CUDA;

  GemmArgs a{};
  a.bits = bits;
  a.perm = r->perm;
  a.inv_perm = r->inv_perm;
  a.block_map = r->block_map;
  a.num_blocks = r->num_blocks;
  a.w = r->w;
  a.ypart = reinterpret_cast<float*>(wsb + L.gemm_ypart);
  a.h_routed = hr;
  a.h_shared = hs;
  a.X = X;
  a.Xh = xh;
  a.Y = Y;
  a.status = status;
  a.T = T;
  a.d = d;
  a.I = I;
  a.k = k;
  a.I_shared = I_shared;
  a.E = E;
  a.num_sms = sm_count();
  a.max_blocks = moe_route_max_blocks(T, E, k, r->block_rows);
  if (a.num_sms <= 0) return MOE_ERR_CUDA;
  if (launch_gemm(a, &mr, shared ? &ms : nullptr, &act, st, pdl) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

moe_status moe_forward(const uint16_t* X, int T, int d, int I, int k, const moe_experts* routed,
                       const moe_experts* shared, int I_shared, const moe_routing* r, uint16_t* Y, void* ws,
                       size_t ws_bytes, moe_stream stream) {
  return forward_impl(X, T, d, I, k, routed, shared, I_shared, r, Y, ws, ws_bytes, stream, nullptr);
}

size_t moe_layer_workspace_bytes(int T, int d, int I, int E, int k, int I_shared) {
  const size_t f = moe_forward_workspace_bytes(T, d, I, E, k, I_shared);
  const size_t r = moe_route_workspace_bytes(T, E, k);
  if (!f || !r) return 0;
  return round256(f) + r;
}

moe_status moe_layer(const float* logits, const uint16_t* X, int T, int d, int I, int k, int block_rows,
                     const moe_experts* routed, const moe_experts* shared, int I_shared, moe_routing* r, uint16_t* Y,
                     void* ws, size_t ws_bytes, moe_stream stream) {
  if (!r || !experts_ok(routed) || T < 0 || k < 1) return MOE_ERR_INVALID_ARG;
  const int E = routed->n_experts;
  if (E > kMaxE || k > kMaxK || k > E) return MOE_ERR_UNSUPPORTED;
  if (block_rows < 1 || block_rows > kMaxBlockRows) return MOE_ERR_UNSUPPORTED;
  if (!r->counts || !r->offsets || !r->block_map || !r->num_blocks) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !r->ids || !r->w || !r->perm || !r->inv_perm)) return MOE_ERR_INVALID_ARG;
  const size_t fbytes = moe_forward_workspace_bytes(T, d, I, E, k, I_shared);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || fbytes == 0 ||
      ws_bytes < moe_layer_workspace_bytes(T, d, I, E, k, I_shared))
    return MOE_ERR_WORKSPACE;
  // One launch when the decode kernel takes the call and can route it itself.
  bool fused = T >= 1 && T <= kGemvMaxT && E <= 256 && decode_supported(T, d, I, I_shared, k);
  if (const char* p = std::getenv("MOE_PATH"))
    if (!std::strcmp(p, "gemm")) fused = false;
  if (fused) {
    r->block_rows = block_rows;
    return forward_impl(X, T, d, I, k, routed, shared, I_shared, r, Y, ws, fbytes, stream, logits);
  }
  // Otherwise the routing kernel, then moe_forward; both report into the first header.
  char* route_ws = static_cast<char*>(ws) + round256(fbytes);
  r->block_rows = block_rows;
  RouteOut o{r->ids, r->w, r->counts, r->offsets, r->perm, r->inv_perm, r->block_map, r->num_blocks};
  const bool pdl = env_flag("MOE_PDL", true);
  if (launch_route(logits, T, E, k, block_rows, o, route_ws, reinterpret_cast<cudaStream_t>(stream), pdl,
                   &static_cast<WsHeader*>(ws)->status) != cudaSuccess)
    return MOE_ERR_CUDA;
  return forward_impl(X, T, d, I, k, routed, shared, I_shared, r, Y, ws, fbytes, stream, nullptr);
}

moe_status moe_layer_x(const uint16_t* X, int T, int d, const uint16_t* W_r, int I, int k, int block_rows,
                       const moe_experts* routed, const moe_experts* shared, int I_shared, float* logits,
                       moe_routing* r, uint16_t* Y, void* ws, size_t ws_bytes, moe_stream stream) {
  // moe_layer's argument checks, before anything is launched
  if (!r || !experts_ok(routed) || T < 0 || k < 1 || d < 64 || d % 64) return MOE_ERR_INVALID_ARG;
  const int E = routed->n_experts;
  if (E > kMaxE || k > kMaxK || k > E) return MOE_ERR_UNSUPPORTED;
  if (block_rows < 1 || block_rows > kMaxBlockRows) return MOE_ERR_UNSUPPORTED;
  if (!r->counts || !r->offsets || !r->block_map || !r->num_blocks) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !r->ids || !r->w || !r->perm || !r->inv_perm)) return MOE_ERR_INVALID_ARG;
  const size_t fbytes = moe_forward_workspace_bytes(T, d, I, E, k, I_shared);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || fbytes == 0 ||
      ws_bytes < moe_layer_workspace_bytes(T, d, I, E, k, I_shared))
    return MOE_ERR_WORKSPACE;
  const moe_status st = moe_router_logits(X, T, d, W_r, E, logits, stream);
  if (st != MOE_OK) return st;
  return moe_layer(logits, X, T, d, I, k, block_rows, routed, shared, I_shared, r, Y, ws, ws_bytes, stream);
}

moe_status moe_check_status(void* ws, moe_stream stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  WsHeader* h = static_cast<WsHeader*>(ws);
  if (cudaMemcpyAsync(&v, &h->status, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    if (cudaMemsetAsync(&h->status, 0, sizeof(uint32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return static_cast<moe_status>(v);
}

}  // extern "C"
