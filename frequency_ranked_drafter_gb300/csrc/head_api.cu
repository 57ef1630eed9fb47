// vt_draft_head / vt_draft_head_ex entry points: argument checks, workspace
// layout, dispatch; vt_draft_noise, the sampler's noise for verification.
#include <cmath>

#include "head_common.cuh"

namespace vt {
namespace {

vt_status draft_head_impl(const char* who, const uint16_t* H, int32_t M,
                          int32_t d, int64_t ldh, const uint16_t* W_high,
                          int32_t V_high, const int32_t* t2f, int32_t k,
                          const HeadOpts& opt, int32_t* out_ids,
                          float* out_probs, float* out_logits, void* ws,
                          size_t ws_bytes, void* stream) {
  const std::string w(who);
  if (!H || !W_high || !out_ids || !out_probs)
    return fail(VT_ERR_INVALID_ARG, w + ": null pointer");
  if (M < 1 || M > 256)
    return fail(VT_ERR_INVALID_ARG, w + ": need 1 <= M <= 256");
  if (d < 8 || d > 16384 || d % 8 != 0)
    return fail(VT_ERR_INVALID_ARG, w + ": need d % 8 == 0 and 8 <= d <= 16384");
  if (ldh < d || ldh % 8 != 0)
    return fail(VT_ERR_INVALID_ARG, w + ": need ldh >= d, ldh % 8 == 0");
  if (V_high < 1) return fail(VT_ERR_INVALID_ARG, w + ": need V_high >= 1");
  if (k < 1 || k > kTopKMax || k > V_high)
    return fail(VT_ERR_INVALID_ARG, w + ": need 1 <= k <= 32 and k <= V_high");
  if (!aligned(H, 16) || !aligned(W_high, 16))
    return fail(VT_ERR_INVALID_ARG, w + ": H, W_high not 16B aligned");
  if (!ws || !aligned(ws, 256) ||
      ws_bytes < vt_draft_head_workspace_size(M, V_high, k))
    return fail(VT_ERR_WORKSPACE, w + ": workspace missing, misaligned or too small");
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (M >= kHeadTcMinM)
    return head_tc(H, M, d, ldh, W_high, V_high, t2f, k, opt, out_ids,
                   out_probs, out_logits, ws, di, s);

  HeadArgs a;
  a.ldh = ldh;
  a.d = d;
  a.W = W_high;
  a.V_high = V_high;
  a.t2f = t2f;
  a.k = k;
  a.opt = opt;
  a.pstride = head_pstride(k, opt.sample != 0);
  a.ticket = static_cast<unsigned*>(ws);
  a.err = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 128);
  a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + kHeadTicketBytes);
  // A few hidden states: the GEMV path.
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

__global__ void draft_noise_kernel(uint64_t seed, uint64_t offset, int m,
                                   const int32_t* ids, int64_t n, float* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = gumbel_noise(seed, offset, m, ids[i]);
}

}  // namespace
}  // namespace vt

extern "C" size_t vt_draft_head_workspace_size(int32_t M, int32_t V_high,
                                               int32_t k) {
  if (M <= 0 || V_high <= 0 || k <= 0) return 0;
  if (M >= vt::kHeadTcMinM) return vt::head_tc_workspace(M, V_high, k);
  return vt::head_gemv_workspace(M, k, /*sample=*/true);
}

extern "C" vt_status vt_draft_head(const uint16_t* H, int32_t M, int32_t d,
                                   int64_t ldh, const uint16_t* W_high,
                                   int32_t V_high, const int32_t* t2f,
                                   int32_t k, int32_t* out_ids,
                                   float* out_probs, float* out_logits,
                                   void* ws, size_t ws_bytes, void* stream) {
  const vt::HeadOpts opt{nullptr, 1.0f, 0, 0, 0};
  return vt::draft_head_impl("vt_draft_head", H, M, d, ldh, W_high, V_high,
                             t2f, k, opt, out_ids, out_probs, out_logits, ws,
                             ws_bytes, stream);
}

namespace vt {

// Checked copy of the public options (NULL = defaults).
static vt_status head_options(const char* who, const vt_head_options* opts,
                              HeadOpts* opt) {
  *opt = HeadOpts{nullptr, 1.0f, 0, 0, 0};
  if (!opts) return VT_OK;
  const std::string w(who);
  if (!(opts->temperature > 0.0f) || !std::isfinite(opts->temperature))
    return fail(VT_ERR_INVALID_ARG, w + ": temperature must be finite and > 0");
  if (opts->mode != VT_HEAD_TOPK && opts->mode != VT_HEAD_SAMPLE)
    return fail(VT_ERR_INVALID_ARG, w + ": unknown mode");
  if (opts->bias_high && !aligned(opts->bias_high, 4))
    return fail(VT_ERR_INVALID_ARG, w + ": bias_high not 4B aligned");
  opt->bias = opts->bias_high;
  opt->tau = opts->temperature;
  opt->sample = opts->mode == VT_HEAD_SAMPLE;
  opt->seed = opts->seed;
  opt->offset = opts->offset;
  return VT_OK;
}

vt_status draft_head_rows(const uint16_t* H, int32_t M, int32_t d, int64_t ldh,
                          const uint16_t* W_high, int32_t V_high,
                          const int32_t* t2f, int32_t k,
                          const vt_head_options* opts, const int32_t* row_ids,
                          int32_t* out_ids, float* out_probs, void* ws,
                          size_t ws_bytes, void* stream) {
  HeadOpts opt;
  vt_status st = head_options("vt_draft_head_sets", opts, &opt);
  if (st != VT_OK) return st;
  opt.row_ids = row_ids;
  return draft_head_impl("vt_draft_head_sets", H, M, d, ldh, W_high, V_high,
                         t2f, k, opt, out_ids, out_probs, nullptr, ws, ws_bytes,
                         stream);
}

}  // namespace vt

extern "C" vt_status vt_draft_head_ex(const uint16_t* H, int32_t M, int32_t d,
                                      int64_t ldh, const uint16_t* W_high,
                                      int32_t V_high, const int32_t* t2f,
                                      int32_t k, const vt_head_options* opts,
                                      int32_t* out_ids, float* out_probs,
                                      float* out_logits, void* ws,
                                      size_t ws_bytes, void* stream) {
  using namespace vt;
  HeadOpts opt;
  vt_status st = head_options("vt_draft_head_ex", opts, &opt);
  if (st != VT_OK) return st;
  return draft_head_impl("vt_draft_head_ex", H, M, d, ldh, W_high, V_high,
                         t2f, k, opt, out_ids, out_probs, out_logits, ws,
                         ws_bytes, stream);
}

extern "C" vt_status vt_draft_noise(uint64_t seed, uint64_t offset, int32_t m,
                                    const int32_t* full_ids, int64_t n,
                                    float* out, void* stream) {
  using namespace vt;
  if (n < 0 || m < 0 || (n > 0 && (!full_ids || !out)))
    return fail(VT_ERR_INVALID_ARG, "vt_draft_noise: bad arguments");
  if (n == 0) return VT_OK;
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)di.num_sms * 8);
  draft_noise_kernel<<<(int)blocks, 256, 0, (cudaStream_t)stream>>>(
      seed, offset, m, full_ids, n, out);
  return launch_status("draft_noise_kernel");
}
