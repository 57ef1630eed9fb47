// Bounds checks of the debug build (nvcc -DVT_CHECKS).
//
// Kernels guard their index-computed global writes (and the reads whose
// index comes from data) with VT_CHECKED(index < size).  In the release build
// the macro is `true` and the guard costs nothing.  In the debug build a
// false condition records its source line in this translation unit's check
// word (the first failure wins) and the guarded access is skipped, so an
// index mistake shows up as a reported line rather than as an access
// outside the buffer; nothing traps.  vt_debug_checks() (vt.h) reads and
// clears every translation unit's word after the work has finished.
#pragma once

#ifdef VT_CHECKS
#include <cuda_runtime.h>

namespace vt {
// Adds a reader of one translation unit's check word (vt_api.cu).
void register_check_word(unsigned (*read_and_clear)());
}  // namespace vt

namespace {
__device__ unsigned vt_check_word;

// The word's value (0: no failure), then 0 again; ~0u if it cannot be read.
unsigned vt_read_check_word() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, vt_check_word, sizeof v) != cudaSuccess) return ~0u;
  if (v && cudaMemcpyToSymbol(vt_check_word, &z, sizeof z) != cudaSuccess) return ~0u;
  return v;
}

struct VtCheckRegistration {
  VtCheckRegistration() { vt::register_check_word(&vt_read_check_word); }
} vt_check_registration;

__device__ __forceinline__ bool vt_check(bool ok, unsigned line) {
  if (!ok) atomicCAS(&vt_check_word, 0u, line);
  return ok;
}
}  // namespace

#define VT_CHECKED(cond) vt_check((cond), __LINE__)
#else
#define VT_CHECKED(cond) true
#endif
