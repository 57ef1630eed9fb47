// vt_draft_q — the full-vocabulary draft distribution of a draft step.
//
// "FR-Spec: Accelerating Large-Vocabulary Language Models via
// Frequency-Ranked Speculative Sampling", Method > Key design: only the
// draft step is trimmed; verification runs the full target model and its
// accept/reject test (rejection sampling) keeps the output distribution
// exactly the target's.  That test compares target and draft probabilities
// over the whole vocabulary, where the trimmed draft gives every dropped id
// probability 0:
//   q[m][f] = exp(s[m][f2t[f]] - max_m) / sum_m   if f2t[f] >= 0,  else 0,
// with s = logit / T over the kept rows (the head's logits, bias included).
//
// Two launches: per row, (max, sum of exp) of s over the V_high logits
// (one CTA per row, online per thread, folded across the block); then the
// fill, eight consecutive ids per thread: f2t and q move in 16-byte vectors
// (when aligned), the kept logits are gathered from L2.  The fill is bound
// by writing q (M * V * 4 bytes).
#include <cmath>

#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kStatThreads = 1024;
constexpr int kFillThreads = 256;
constexpr int kFillIds = 8;  // ids per thread

// Folds (m2, s2) into (m, s), pairs of (max, sum of exp(x - max)); empty
// pairs (-inf, 0) are neutral.
__device__ __forceinline__ void fold(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  s = (s > 0.f ? s * expf(m - M) : 0.f) + (s2 > 0.f ? s2 * expf(m2 - M) : 0.f);
  m = M;
}

__global__ void __launch_bounds__(kStatThreads)
    q_stats_kernel(const float* __restrict__ logits, int V_high, float inv_tau,
                   float2* __restrict__ stats) {
  __shared__ float wm[kStatThreads / 32], wsum[kStatThreads / 32];
  const float* row = logits + (size_t)blockIdx.x * V_high;
  float m = -INFINITY, s = 0.f;
  for (int i = threadIdx.x; i < V_high; i += kStatThreads) {
    const float x = __ldcg(row + i) * inv_tau;
    if (x > m) {
      s = (s > 0.f ? s * expf(m - x) : 0.f) + 1.f;
      m = x;
    } else {
      s += expf(x - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(~0u, m, o);
    const float s2 = __shfl_xor_sync(~0u, s, o);
    fold(m, s, m2, s2);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { wm[warp] = m; wsum[warp] = s; }
  __syncthreads();
  if (warp == 0) {
    m = wm[lane];
    s = wsum[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(~0u, m, o);
      const float s2 = __shfl_xor_sync(~0u, s, o);
      fold(m, s, m2, s2);
    }
    if (lane == 0) stats[blockIdx.x] = make_float2(m, s);
  }
}

__global__ void __launch_bounds__(kFillThreads)
    q_fill_kernel(const float* __restrict__ logits, int V_high,
                  const int32_t* __restrict__ f2t, int V, float inv_tau,
                  const float2* __restrict__ stats, float* __restrict__ q,
                  bool vec) {
  const int m = blockIdx.y;
  const float2 st = stats[m];
  const float inv_sum = 1.f / st.y;
  const float* row = logits + (size_t)m * V_high;
  float* qm = q + (size_t)m * V;
  const int f0 = (blockIdx.x * kFillThreads + threadIdx.x) * kFillIds;
  if (f0 >= V) return;
  int idx[kFillIds];
  if (vec && f0 + kFillIds <= V) {
    if (f2t) {
      const int4 a = __ldg(reinterpret_cast<const int4*>(f2t + f0));
      const int4 b = __ldg(reinterpret_cast<const int4*>(f2t + f0) + 1);
      idx[0] = a.x; idx[1] = a.y; idx[2] = a.z; idx[3] = a.w;
      idx[4] = b.x; idx[5] = b.y; idx[6] = b.z; idx[7] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < kFillIds; ++j) idx[j] = f0 + j;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kFillIds; ++j)
      idx[j] = f0 + j < V ? (f2t ? __ldg(f2t + f0 + j) : f0 + j) : -1;
  }
  float v[kFillIds];
#pragma unroll
  for (int j = 0; j < kFillIds; ++j)
    v[j] = (idx[j] >= 0 && idx[j] < V_high) ? __ldcg(row + idx[j]) : -INFINITY;
#pragma unroll
  for (int j = 0; j < kFillIds; ++j)
    v[j] = v[j] == -INFINITY ? 0.f : expf(v[j] * inv_tau - st.x) * inv_sum;
  if (vec && f0 + kFillIds <= V) {
    float4* dst = reinterpret_cast<float4*>(qm + f0);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
#pragma unroll
    for (int j = 0; j < kFillIds; ++j)
      if (f0 + j < V) qm[f0 + j] = v[j];
  }
}

}  // namespace
}  // namespace vt

extern "C" size_t vt_draft_q_workspace_size(int32_t M) {
  return M > 0 ? (size_t)M * 8 : 0;
}

extern "C" vt_status vt_draft_q(const float* logits, int32_t M, int32_t V_high,
                                const int32_t* f2t, int32_t V,
                                float temperature, float* q, void* ws,
                                size_t ws_bytes, void* stream) {
  using namespace vt;
  if (!logits || !q) return fail(VT_ERR_INVALID_ARG, "vt_draft_q: null pointer");
  if (M < 1 || M > 65535 || V_high < 1 || V < V_high)
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_q: need 1 <= M <= 65535, V_high >= 1, V >= V_high");
  if (!f2t && V != V_high)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_q: f2t = NULL needs V == V_high");
  if (!(temperature > 0.0f) || !std::isfinite(temperature))
    return fail(VT_ERR_INVALID_ARG, "vt_draft_q: temperature must be finite and > 0");
  if (!aligned(logits, 4) || !aligned(q, 4) || (f2t && !aligned(f2t, 4)))
    return fail(VT_ERR_INVALID_ARG, "vt_draft_q: logits, q, f2t not 4B aligned");
  const float* l_end = logits + (size_t)M * V_high;
  const float* q_end = q + (size_t)M * V;
  if (logits < q_end && q < l_end)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_q: q overlaps logits");
  if (!ws || !aligned(ws, 8) || ws_bytes < vt_draft_q_workspace_size(M))
    return fail(VT_ERR_WORKSPACE, "vt_draft_q: workspace missing, misaligned or too small");
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const float inv_tau = 1.0f / temperature;
  float2* stats = static_cast<float2*>(ws);
  q_stats_kernel<<<M, kStatThreads, 0, s>>>(logits, V_high, inv_tau, stats);
  vt_status st = launch_status("q_stats_kernel");
  if (st != VT_OK) return st;
  // 16-byte vectors when every row of q and f2t starts 16-byte aligned
  const bool vec = (V % 4 == 0) && aligned(q, 16) && (!f2t || aligned(f2t, 16));
  const int per_block = kFillThreads * kFillIds;
  dim3 grid((V + per_block - 1) / per_block, M);
  q_fill_kernel<<<grid, kFillThreads, 0, s>>>(logits, V_high, f2t, V, inv_tau,
                                              stats, q, vec);
  return launch_status("q_fill_kernel");
}
