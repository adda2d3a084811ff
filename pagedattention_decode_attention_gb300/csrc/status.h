// Host-side error reporting shared by every translation unit of the library.
#pragma once

#include <cstdint>

namespace pa {

// Records a printf-style message for pa_last_error() on this thread and
// returns `code`.
int fail(int code, const char* fmt, ...);

// Bits of the device status word (one 32-bit word per device).
constexpr unsigned kStatusBounds = 1u;   // clamped or skipped an out-of-range index
constexpr unsigned kStatusTimeout = 2u;  // a bounded device-side wait ran out
constexpr unsigned kStatusPlan = 4u;     // a decode run found no matching plan in its workspace

// Device address of this device's status word (looked up once per device).
// Returns nullptr and records an error when the CUDA runtime fails.
unsigned* device_status_word();

}  // namespace pa
