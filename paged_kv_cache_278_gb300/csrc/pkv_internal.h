// pkv_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <stdint.h>

namespace pkv_internal {

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline bool aligned16(const void *p) { return aligned(p, 16); }

// Each kernel translation unit owns one device error word; these read it for
// the current device and reset it to zero.  Return PKV_OK or PKV_ERR_CUDA.
int append_take_error(int *code);
int decode_take_error(int *code);

}  // namespace pkv_internal
