// Status strings, error recording and the device-info cache of the C ABI.
#include <mutex>
#include <set>
#include <string>
#include <utility>

#include <vector>

#include "vt_common.cuh"

namespace vt {

// Readers of the translation units' check words (debug builds only; each
// unit registers at load time).
static std::vector<unsigned (*)()>& check_readers() {
  static std::vector<unsigned (*)()> readers;
  return readers;
}

void register_check_word(unsigned (*read_and_clear)()) {
  check_readers().push_back(read_and_clear);
}

static thread_local std::string g_last_error;

vt_status fail(vt_status s, const std::string& why) {
  g_last_error = why;
  return s;
}

bool current_device(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    g_last_error = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
    return false;
  }
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& di = cache[dev];
  if (di.device != dev) {
    DeviceInfo t;
    t.device = dev;
    if (cudaDeviceGetAttribute(&t.num_sms, cudaDevAttrMultiProcessorCount,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.max_smem_optin,
                               cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.cc_major, cudaDevAttrComputeCapabilityMajor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.cc_minor, cudaDevAttrComputeCapabilityMinor,
                               dev) != cudaSuccess) {
      g_last_error = "cudaDeviceGetAttribute failed";
      return false;
    }
    di = t;
  }
  *out = di;
  return true;
}

bool allow_max_smem_impl(const void* kernel, const DeviceInfo& di) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, di.device);
  if (done.count(key)) return true;
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             di.max_smem_optin - (int)fa.sharedSizeBytes);
  if (e != cudaSuccess) {
    g_last_error = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return false;
  }
  done.insert(key);
  return true;
}

vt_status launch_status(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(VT_ERR_CUDA,
                std::string(what) + ": " + cudaGetErrorString(e));
  return VT_OK;
}

}  // namespace vt

extern "C" {

const char* vt_status_string(int status) {
  switch (status) {
    case VT_OK: return "VT_OK";
    case VT_ERR_INVALID_ARG: return "VT_ERR_INVALID_ARG";
    case VT_ERR_CUDA: return "VT_ERR_CUDA";
    case VT_ERR_UNSUPPORTED: return "VT_ERR_UNSUPPORTED";
    case VT_ERR_WORKSPACE: return "VT_ERR_WORKSPACE";
    case VT_ERR_TIMEOUT: return "VT_ERR_TIMEOUT";
    default: return "VT_ERR_UNKNOWN";
  }
}

const char* vt_last_error(void) { return vt::g_last_error.c_str(); }

int vt_version(void) { return 102; }

int vt_debug_build(void) {
#ifdef VT_CHECKS
  return 1;
#else
  return 0;
#endif
}

int vt_debug_checks(void) {
  int first = 0;
  for (auto read : vt::check_readers()) {
    const unsigned v = read();
    if (v == ~0u) return -1;
    if (v && !first) first = (int)v;
  }
  return first;
}

size_t vt_workspace_size(int32_t op, int32_t M, int32_t n, int32_t k) {
  switch (op) {
    case VT_OP_COUNT: return vt_count_tokens_workspace_size(n);
    case VT_OP_SELECT: return vt_select_vocab_workspace_size(n);
    case VT_OP_HEAD: return vt_draft_head_workspace_size(M, n, k);
    case VT_OP_Q: return vt_draft_q_workspace_size(M);
    default: return 0;
  }
}

}  // extern "C"
