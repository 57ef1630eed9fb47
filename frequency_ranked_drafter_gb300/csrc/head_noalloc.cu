// vt_draft_head_noalloc — the draft head for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they run a draft step: code running inside a CUDA stream
// capture that must not add allocation nodes, real-time or embedded hosts
// that forbid allocation after start-up, and plugins that live inside
// another framework's memory pool and may not create allocations of their
// own.  For them this file keeps the draft head's scratch (the grid-wide
// arrival counters and every CTA's partial results) in one file-scope
// device array, so a call needs no workspace argument and allocates
// nothing.
//
// The array has a fixed size (kNoAllocScratchBytes, 1 MiB) and every GPU
// that loads the library holds one copy until the process exits.  All
// calls on a device share that copy: two calls that overlap on the GPU
// (different streams, no ordering between them) race on it and give wrong
// results; calls on one stream, or otherwise ordered, are fine.
//
// The first call on each device sets the array up: with that device
// current it looks up the array's device address (in host code the
// array's name is only a host-side stand-in, never a device pointer) and
// zero-fills the arrival counters with a synchronous cudaMemset.  Make that
// first call before starting any stream capture.  Later calls reuse the
// cached address, and every completed call leaves the counters at zero.
#include <mutex>
#include <string>

#include "head_common.cuh"

namespace vt {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) unsigned char g_head_scratch[kNoAllocScratchBytes];

// Device address of g_head_scratch for the current device, set up once per
// device.  Returns nullptr (and records why) on failure.
void* noalloc_scratch(const DeviceInfo& di) {
  static std::mutex mu;
  static void* addr[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (di.device < 0 || di.device >= 64) {
    fail(VT_ERR_UNSUPPORTED, "vt_draft_head_noalloc: device index >= 64");
    return nullptr;
  }
  if (addr[di.device]) return addr[di.device];
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_head_scratch);
  if (e != cudaSuccess || p == nullptr) {
    fail(VT_ERR_CUDA, std::string("vt_draft_head_noalloc: cudaGetSymbolAddress: ") +
                          cudaGetErrorString(e));
    return nullptr;
  }
  // the arrival counters must start at zero; calls leave them at zero
  e = cudaMemset(p, 0, kHeadTicketBytes);
  if (e != cudaSuccess) {
    fail(VT_ERR_CUDA, std::string("vt_draft_head_noalloc: cudaMemset: ") +
                          cudaGetErrorString(e));
    return nullptr;
  }
  addr[di.device] = p;
  return p;
}

}  // namespace
}  // namespace vt

extern "C" vt_status vt_draft_head_noalloc(const uint16_t* H, int32_t M,
                                           int32_t d, int64_t ldh,
                                           const uint16_t* W_high,
                                           int32_t V_high, const int32_t* t2f,
                                           int32_t k, int32_t* out_ids,
                                           float* out_probs, float* out_logits,
                                           void* stream) {
  using namespace vt;
  if (!H || !W_high || !out_ids || !out_probs)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head_noalloc: null pointer");
  if (M < 1 || M > 256)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head_noalloc: need 1 <= M <= 256");
  if (d < 8 || d > 16384 || d % 8 != 0)
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_head_noalloc: need d % 8 == 0 and 8 <= d <= 16384");
  if (ldh < d || ldh % 8 != 0)
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_head_noalloc: need ldh >= d, ldh % 8 == 0");
  if (V_high < 1)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head_noalloc: need V_high >= 1");
  if (k < 1 || k > kTopKMax || k > V_high)
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_head_noalloc: need 1 <= k <= 32 and k <= V_high");
  if (!aligned(H, 16) || !aligned(W_high, 16))
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_head_noalloc: H, W_high not 16B aligned");
  // Hidden states are processed four at a time by the GEMV kernel, each
  // group reusing the same scratch, so the need depends on min(M, 4) and k.
  const size_t need = head_gemv_workspace(std::min(M, 4), k, /*sample=*/false);
  if (need > kNoAllocScratchBytes)
    return fail(VT_ERR_UNSUPPORTED,
                "vt_draft_head_noalloc: needs " + std::to_string(need) +
                    " bytes of scratch but has " +
                    std::to_string(kNoAllocScratchBytes) +
                    " (reduce k, or use vt_draft_head with a workspace)");
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  void* scratch = noalloc_scratch(di);
  if (!scratch) return VT_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;

  HeadArgs a;
  a.ldh = ldh;
  a.d = d;
  a.W = W_high;
  a.V_high = V_high;
  a.t2f = t2f;
  a.k = k;
  a.pstride = head_pstride(k, false);
  a.opt = HeadOpts{nullptr, 1.0f, 0, 0, 0};
  a.ticket = static_cast<unsigned*>(scratch);
  a.err = reinterpret_cast<unsigned*>(static_cast<char*>(scratch) + 128);
  a.part = reinterpret_cast<float*>(static_cast<char*>(scratch) +
                                    kHeadTicketBytes);
  for (int m0 = 0; m0 < M; m0 += 4) {
    a.M = std::min(4, M - m0);
    a.m_base = m0;
    a.H = H + (int64_t)m0 * ldh;
    a.out_ids = out_ids + (int64_t)m0 * k;
    a.out_probs = out_probs + (int64_t)m0 * k;
    a.out_logits = out_logits ? out_logits + (int64_t)m0 * V_high : nullptr;
    vt_status st = head_gemv(a, di, s);
    if (st != VT_OK) return st;
  }
  return VT_OK;
}
