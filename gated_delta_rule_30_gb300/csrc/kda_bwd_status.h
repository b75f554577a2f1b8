// kda_bwd_status.h -- the backward pass's own bit of the library status word
// (kda_device_status; the other bits are in kda_internal.h).
#pragma once

namespace kda {

// a low-memory kda_bwd call found no free replay slot (outputs undefined)
constexpr int kStatusScratch = 8;

}  // namespace kda
