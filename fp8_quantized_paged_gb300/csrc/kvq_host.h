// kvq_host.h -- host-side helpers shared by the entry points of libkvq.
#pragma once

#include <stdint.h>

namespace kvq {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device (cached per device); 0 if no device.
int device_sm_count();

}  // namespace kvq
