// Status codes and workspace header shared by the host boundary and the kernels.
#pragma once

#include <cstdint>

#include "moe.h"

namespace bm {

// Every workspace starts with this header (256 bytes, so what follows stays
// 256-byte aligned).
struct WsHeader {
  uint32_t status;     // first device-side error (moe_status), 0 = none
  uint32_t ticket;     // arrival counter of the routing kernel; reset by its last CTA
  uint32_t route_done;  // routing kernel (grid-synchronised mode): CTAs that have finished
  uint32_t dec_gen;     // decode kernel: calls so far; call g counts its barrier arrivals in dec_count[g % 2]
  uint32_t dec_count[2];
  uint32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "workspace header must be 256 bytes");

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxBlockRows = 128;
constexpr int kRouteTokensPerCta = 32;
constexpr int kGemvMaxT = 4;

}  // namespace bm
