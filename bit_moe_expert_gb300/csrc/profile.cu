// Per-kernel event timing (include/moe_profile.h).  Off by default; when on,
// each launch is bracketed by two events on its own stream.
#include <cuda_runtime.h>

#include <vector>

#include "kernels.h"
#include "moe_profile.h"

namespace bm {
namespace {

const char* const kNames[kKernelKinds] = {"route", "decode", "router", "x_gather",
                                          "gemm_gateup", "gemm_down", "combine", "prepack",
                                          "topk_wide"};

struct Pending {
  int id;
  cudaEvent_t start, stop;
};

bool g_on = false;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free;
double g_total_ms[kKernelKinds] = {0};
long long g_count[kKernelKinds] = {0};
cudaEvent_t g_open_start = nullptr;

cudaEvent_t take_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

bool drain() {
  bool ok = true;
  for (const Pending& p : g_pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(p.stop) != cudaSuccess || cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess)
      ok = false;
    else {
      g_total_ms[p.id] += ms;
      g_count[p.id] += 1;
    }
    g_free.push_back(p.start);
    g_free.push_back(p.stop);
  }
  g_pending.clear();
  return ok;
}

}  // namespace

void timer_begin(int id, cudaStream_t s) {
  (void)id;
  if (!g_on) return;
  g_open_start = take_event();
  if (g_open_start) cudaEventRecord(g_open_start, s);
}

void timer_end(int id, cudaStream_t s) {
  if (!g_on || !g_open_start) return;
  cudaEvent_t stop = take_event();
  if (!stop) return;
  cudaEventRecord(stop, s);
  g_pending.push_back(Pending{id, g_open_start, stop});
  g_open_start = nullptr;
  if (g_pending.size() >= 4096) drain();
}

}  // namespace bm

using namespace bm;

extern "C" {

int moe_profile_enable(int on) {
  const int prev = g_on ? 1 : 0;
  g_on = on != 0;
  return prev;
}

int moe_profile_kernel_count(void) { return kKernelKinds; }

const char* moe_profile_kernel_name(int id) { return (id >= 0 && id < kKernelKinds) ? kNames[id] : nullptr; }

moe_status moe_profile_read(int id, double* total_ms, long long* launches) {
  if (id < 0 || id >= kKernelKinds || !total_ms || !launches) return MOE_ERR_INVALID_ARG;
  const bool ok = drain();
  *total_ms = g_total_ms[id];
  *launches = g_count[id];
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

void moe_profile_reset(void) {
  drain();
  for (int i = 0; i < kKernelKinds; ++i) {
    g_total_ms[i] = 0.0;
    g_count[i] = 0;
  }
}

}  // extern "C"

extern "C" moe_status moe_debug_decode(long long wait_limit_cycles, int drop_cta) {
  if (drop_cta < -1) return MOE_ERR_INVALID_ARG;
  return bm::decode_debug(wait_limit_cycles, drop_cta) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
