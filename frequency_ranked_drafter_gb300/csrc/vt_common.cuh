// Shared device/host helpers of the GB300 library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <string>
#include <utility>

#include "vt.h"

namespace vt {

// ---------------------------------------------------------------- host side

// Records the reason for a non-OK status (thread-local, read by
// vt_last_error) and returns the status.
vt_status fail(vt_status s, const std::string& why);

// Per-device facts cached on first use.
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int max_smem_optin = 0;  // bytes per block
  int cc_major = 0, cc_minor = 0;
};
// Info for the current device; returns false (and records why) on failure.
bool current_device(DeviceInfo* out);

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Maps the result of a kernel launch to a status.
vt_status launch_status(const char* what);

// Launches `kernel` as a programmatic dependent of the work ahead of it in
// stream `s` (see grid_dependency_wait below): the kernel may start while
// the previous kernel finishes and must wait before reading its results.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block,
                             size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Opts `kernel` in to the device's full dynamic shared memory, once per
// (kernel, device), so later calls (including ones under stream capture)
// make no attribute call.  Returns false (and records why) on failure.
bool allow_max_smem_impl(const void* kernel, const DeviceInfo& di);
template <typename Kernel>
bool allow_max_smem(Kernel kernel, const DeviceInfo& di) {
  return allow_max_smem_impl(reinterpret_cast<const void*>(kernel), di);
}

// ------------------------------------------------------------- device side

// bf16 bit pairs packed in a 32-bit word -> the two fp32 values (exact).
__device__ __forceinline__ float bf16lo(uint32_t x) {
  return __uint_as_float(x << 16);
}
__device__ __forceinline__ float bf16hi(uint32_t x) {
  return __uint_as_float(x & 0xffff0000u);
}

// 16-byte streaming load of read-once data: not kept in L1, evict-first in
// L2, with a 256-byte L2 prefetch hint.
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ int4 ld_stream_i4(const void* p) {
  int4 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::256B.v4.s32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream_u4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Programmatic dependent launch (PTX griddepcontrol).  A kernel launched
// with the programmatic-serialization attribute may start before the kernel
// ahead of it in the stream has ended; it must read nothing that kernel may
// write before grid_dependency_wait(), which returns once that kernel has
// completed and its writes are visible (at once when launched normally).
// grid_launch_dependents() lets the next such kernel start early.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Asks L2 to fetch `bytes` (a multiple of 16) from a 16-byte-aligned global
// address.  A hint: it returns nothing and orders nothing, so it is safe even
// before grid_dependency_wait() (the loads that use the data come later and
// read L2, where every store lands).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ unsigned lane_id() {
  unsigned r;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(r));
  return r;
}

}  // namespace vt
