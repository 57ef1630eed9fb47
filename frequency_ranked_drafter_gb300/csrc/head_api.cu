// vt_draft_head entry point: argument checks, workspace layout, dispatch.
#include "head_common.cuh"

extern "C" size_t vt_draft_head_workspace_size(int32_t M, int32_t V_high,
                                               int32_t k) {
  if (M <= 0 || V_high <= 0 || k <= 0) return 0;
  if (M >= vt::kHeadTcMinM) return vt::head_tc_workspace(M, V_high, k);
  return vt::head_gemv_workspace(M, k);
}

extern "C" vt_status vt_draft_head(const uint16_t* H, int32_t M, int32_t d,
                                   int64_t ldh, const uint16_t* W_high,
                                   int32_t V_high, const int32_t* t2f,
                                   int32_t k, int32_t* out_ids,
                                   float* out_probs, float* out_logits,
                                   void* ws, size_t ws_bytes, void* stream) {
  using namespace vt;
  if (!H || !W_high || !out_ids || !out_probs)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head: null pointer");
  if (M < 1 || M > 256)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head: need 1 <= M <= 256");
  if (d < 8 || d > 16384 || d % 8 != 0)
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_head: need d % 8 == 0 and 8 <= d <= 16384");
  if (ldh < d || ldh % 8 != 0)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head: need ldh >= d, ldh % 8 == 0");
  if (V_high < 1)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head: need V_high >= 1");
  if (k < 1 || k > kTopKMax || k > V_high)
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_head: need 1 <= k <= 32 and k <= V_high");
  if (!aligned(H, 16) || !aligned(W_high, 16))
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head: H, W_high not 16B aligned");
  if (!ws || !aligned(ws, 256) ||
      ws_bytes < vt_draft_head_workspace_size(M, V_high, k))
    return fail(VT_ERR_WORKSPACE,
                "vt_draft_head: workspace missing, misaligned or too small");
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (M >= kHeadTcMinM)
    return head_tc(H, M, d, ldh, W_high, V_high, t2f, k, out_ids, out_probs,
                   out_logits, ws, di, s);

  HeadArgs a;
  a.ldh = ldh;
  a.d = d;
  a.W = W_high;
  a.V_high = V_high;
  a.t2f = t2f;
  a.k = k;
  a.pstride = head_pstride(k);
  a.ticket = static_cast<unsigned*>(ws);
  a.err = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 128);
  a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + kHeadTicketBytes);
  // A few hidden states: the GEMV path.
  for (int m0 = 0; m0 < M; m0 += 4) {
    a.M = std::min(4, M - m0);
    a.H = H + (int64_t)m0 * ldh;
    a.out_ids = out_ids + (int64_t)m0 * k;
    a.out_probs = out_probs + (int64_t)m0 * k;
    a.out_logits = out_logits ? out_logits + (int64_t)m0 * V_high : nullptr;
    vt_status st = head_gemv(a, di, s);
    if (st != VT_OK) return st;
  }
  return VT_OK;
}
