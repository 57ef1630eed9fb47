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
// When a row of logits fits in shared memory (V_high <= ~56K): one kernel,
// each CTA staging its row there (q_row_kernel).  Otherwise two launches:
// per row, (max, sum of exp) of s (one CTA per row, batched loads), then the
// fill, eight consecutive ids for four rows per thread with the kept logits
// gathered from L2.  Both are bound by writing q (M * V * 4 bytes).
#include <cmath>

#include "vt_checks.cuh"
#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kStatThreads = 1024;
constexpr int kFillThreads = 256;
constexpr int kFillIds = 8;  // ids per thread
constexpr int kFillRows = 4;  // rows per thread

// Folds (m2, s2) into (m, s), pairs of (max, sum of exp(x - max)); empty
// pairs (-inf, 0) are neutral.
__device__ __forceinline__ void fold(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  s = (s > 0.f ? s * expf(m - M) : 0.f) + (s2 > 0.f ? s2 * expf(m2 - M) : 0.f);
  m = M;
}

// Row statistics: each thread folds its values of the row online; the
// loads go out eight 16-byte vectors at a time (or eight scalars when the
// row is not 16-byte aligned), so one L2 round trip serves 32 values.
__global__ void __launch_bounds__(kStatThreads)
    q_stats_kernel(const float* __restrict__ logits, int V_high, float inv_tau,
                   float2* __restrict__ stats, bool vec) {
  __shared__ float wm[kStatThreads / 32], wsum[kStatThreads / 32];
  const float* row = logits + (size_t)blockIdx.x * V_high;
  float m = -INFINITY, s = 0.f;
  auto add = [&](float x) {
    if (x == -INFINITY) return;  // padding
    x *= inv_tau;
    if (x > m) {
      s = (s > 0.f ? s * expf(m - x) : 0.f) + 1.f;
      m = x;
    } else {
      s += expf(x - m);
    }
  };
  constexpr int kBatch = 8;
  if (vec) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = V_high / 4;
    for (int base = 0; base < n4; base += kStatThreads * kBatch) {
      float4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kStatThreads + threadIdx.x;
        v[j] = i < n4 ? __ldcg(r4 + i)
                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        add(v[j].x); add(v[j].y); add(v[j].z); add(v[j].w);
      }
    }
  } else {
    for (int base = 0; base < V_high; base += kStatThreads * kBatch) {
      float v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kStatThreads + threadIdx.x;
        v[j] = i < V_high ? __ldcg(row + i) : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) add(v[j]);
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

// Fill: a thread owns eight consecutive full ids for kFillRows rows: one
// read of their f2t entries serves every row; the kept logits are gathered
// from L2 and each row's q segment is written with two 16-byte stores (or
// scalars at a ragged end / unaligned rows).
__global__ void __launch_bounds__(kFillThreads)
    q_fill_kernel(const float* __restrict__ logits, int M, int V_high,
                  const int32_t* __restrict__ f2t, int V, float inv_tau,
                  const float2* __restrict__ stats, float* __restrict__ q,
                  bool vec) {
  const int f0 = (blockIdx.x * kFillThreads + threadIdx.x) * kFillIds;
  if (f0 >= V) return;
  const bool full = vec && f0 + kFillIds <= V;
  int idx[kFillIds];
  if (full && f2t) {
    const int4 a = __ldg(reinterpret_cast<const int4*>(f2t + f0));
    const int4 b = __ldg(reinterpret_cast<const int4*>(f2t + f0) + 1);
    idx[0] = a.x; idx[1] = a.y; idx[2] = a.z; idx[3] = a.w;
    idx[4] = b.x; idx[5] = b.y; idx[6] = b.z; idx[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < kFillIds; ++j)
      idx[j] = f0 + j < V ? (f2t ? __ldg(f2t + f0 + j) : f0 + j) : -1;
  }
  const int m0 = blockIdx.y * kFillRows;
  float v[kFillRows][kFillIds];
#pragma unroll
  for (int r = 0; r < kFillRows; ++r) {
    const int m = min(m0 + r, M - 1);
    const float* row = logits + (size_t)m * V_high;
#pragma unroll
    for (int j = 0; j < kFillIds; ++j)
      v[r][j] = (idx[j] >= 0 && idx[j] < V_high) ? __ldcg(row + idx[j]) : -INFINITY;
  }
#pragma unroll
  for (int r = 0; r < kFillRows; ++r) {
    const int m = m0 + r;
    if (m >= M) break;
    const float2 st = stats[m];
    const float inv_sum = 1.f / st.y;
    float o[kFillIds];
#pragma unroll
    for (int j = 0; j < kFillIds; ++j)
      o[j] = v[r][j] == -INFINITY ? 0.f : expf(v[r][j] * inv_tau - st.x) * inv_sum;
    float* qm = q + (size_t)m * V;
    if (full) {
      float4* dst = reinterpret_cast<float4*>(qm + f0);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    } else {
#pragma unroll
      for (int j = 0; j < kFillIds; ++j)
        if (f0 + j < V) qm[f0 + j] = o[j];
    }
  }
}

// One kernel when a row of logits fits in shared memory: grid (P, M); every
// CTA of row m stages the row's V_high values of logit / T in shared memory
// (coalesced 16-byte loads) taking their maximum on the way, sums
// exp(s - max) from shared memory in a second pass (no branch and one
// exponential per value, where an online fold needed a compare and up to
// two), then fills its 1/P of q[m], the kept values gathered from shared
// memory (no L2 sector per gathered value), f2t loads and q stores both
// 512 contiguous bytes per warp instruction.
// Exponentials use the fast hardware form (relative error about 1e-6 here,
// far inside the 1e-4 bound on q).
constexpr int kRowQThreads = 1024;

// Stages row m's logit / T in srow and returns (max, 1 / sum of exp(s -
// max)) to every thread of the CTA.
__device__ __forceinline__ float2 stage_row_stats(const float* __restrict__ row,
                                                  int V_high, float inv_tau,
                                                  float* srow) {
  __shared__ float wm[kRowQThreads / 32], wsum[kRowQThreads / 32];
  __shared__ float2 st_all;
  float mm = -INFINITY;
  if ((V_high & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    float4* s4 = reinterpret_cast<float4*>(srow);
    const int n4 = V_high / 4;
    constexpr int kBatch = 8;  // loads in flight per thread
    for (int base = 0; base < n4; base += kRowQThreads * kBatch) {
      float4 x[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kRowQThreads + threadIdx.x;
        if (i < n4) x[j] = __ldcg(r4 + i);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kRowQThreads + threadIdx.x;
        if (i < n4) {
          float4 y = x[j];
          y.x *= inv_tau; y.y *= inv_tau; y.z *= inv_tau; y.w *= inv_tau;
          s4[i] = y;
          mm = fmaxf(mm, fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w)));
        }
      }
    }
  } else {
    for (int i = threadIdx.x; i < V_high; i += kRowQThreads) {
      const float x = __ldcg(row + i) * inv_tau;
      srow[i] = x;
      mm = fmaxf(mm, x);
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(~0u, mm, o));
  if (lane == 0) wm[warp] = mm;
  __syncthreads();  // also publishes the staged row
  mm = wm[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(~0u, mm, o));
  float ss = 0.f;
  for (int i = threadIdx.x; i < V_high; i += kRowQThreads) ss += __expf(srow[i] - mm);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(~0u, ss, o);
  if (lane == 0) wsum[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    ss = wsum[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(~0u, ss, o);
    if (lane == 0) st_all = make_float2(mm, 1.f / ss);
  }
  __syncthreads();
  return st_all;
}

// With at most two parts per row (`pre`: each CTA fills half of q's row or
// all of it), the staged row is turned into probabilities once, exp(s - max) /
// sum in place, and the fill only gathers them: the same values, and the
// exponentials leave the fill loop (M = 60: 12.6 -> 11.7 us); with many
// parts per row the extra pass over the whole row costs more than it saves
// (M = 1: 5.2 -> 6.1 us), and the fill computes them.
__global__ void __launch_bounds__(kRowQThreads, 1)
    q_row_kernel(const float* __restrict__ logits, int V_high,
                 const int32_t* __restrict__ f2t, int V, float inv_tau,
                 float* __restrict__ q, int span, bool vec, bool pre) {
  extern __shared__ __align__(16) float srow[];  // [V_high] logit / T
  const int m = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* row = logits + (size_t)m * V_high;
  const int f_begin = blockIdx.x * span, f_end = min(V, f_begin + span);
  if (!VT_CHECKED(f_begin < V)) return;  // the grid covers V exactly
  // A warp's step covers 32 * kFillIds consecutive ids; lane l takes the
  // four-id chunks at 4 l and 4 l + 128, so every f2t load and q store of
  // the warp is 512 contiguous bytes.  The first step's f2t entries are
  // requested before the row is staged, each next step's before the current
  // one is written.
  static_assert(kFillIds == 8, "two chunks of four ids per lane");
  auto load_idx = [&](int fw, int (&idx)[kFillIds]) {
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int f = fw + 128 * v + 4 * lane;
      if (vec && f2t && f + 4 <= f_end) {
        const int4 x = __ldg(reinterpret_cast<const int4*>(f2t + f));
        idx[4 * v] = x.x; idx[4 * v + 1] = x.y; idx[4 * v + 2] = x.z; idx[4 * v + 3] = x.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          idx[4 * v + j] = f + j < f_end ? (f2t ? __ldg(f2t + f + j) : f + j) : -1;
      }
    }
  };
  constexpr int kStep = kRowQThreads * kFillIds;
  int idx[kFillIds];
  int fw = f_begin + warp * 32 * kFillIds;
  if (fw < f_end) load_idx(fw, idx);
  const float2 st = stage_row_stats(row, V_high, inv_tau, srow);
  const float mx = st.x, inv_sum = st.y;
  if (pre) {
    for (int i = threadIdx.x; i < V_high; i += kRowQThreads)
      srow[i] = __expf(srow[i] - mx) * inv_sum;
    __syncthreads();
  }
  float* qm = q + (size_t)m * V;
  for (; fw < f_end; fw += kStep) {
    int nidx[kFillIds];
    if (fw + kStep < f_end) load_idx(fw + kStep, nidx);
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int f = fw + 128 * v + 4 * lane;
      float o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ix = idx[4 * v + j];
        o[j] = (unsigned)ix >= (unsigned)V_high ? 0.f
               : pre ? srow[ix] : __expf(srow[ix] - mx) * inv_sum;
      }
      if (vec && f + 4 <= f_end) {
        *reinterpret_cast<float4*>(qm + f) = make_float4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (f + j < f_end) qm[f + j] = o[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kFillIds; ++j) idx[j] = nidx[j];
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
  // 16-byte vectors when every row of q and f2t starts 16-byte aligned
  const bool vec = (V % 4 == 0) && aligned(q, 16) && (!f2t || aligned(f2t, 16));
  const size_t row_bytes = (size_t)V_high * sizeof(float);
  if (row_bytes + 1024 <= (size_t)di.max_smem_optin) {
    // P parts per row: one wave of CTAs (one fits an SM), at least 1024 ids
    // a part, spans that are whole multiples of the vector width
    const int want = std::max(1, di.num_sms / M);
    const int per_part_min = 1024;
    const int P = std::max(1, std::min(want, (V + per_part_min - 1) / per_part_min));
    int span = (V + P - 1) / P;
    span = (span + kFillIds - 1) / kFillIds * kFillIds;
    const dim3 grid((V + span - 1) / span, M);
    if (!allow_max_smem(q_row_kernel, di)) return VT_ERR_CUDA;
    q_row_kernel<<<grid, kRowQThreads, row_bytes, s>>>(logits, V_high, f2t, V,
                                                       inv_tau, q, span, vec,
                                                       grid.x <= 2);
    return launch_status("q_row_kernel");
  }
  float2* stats = static_cast<float2*>(ws);
  const bool vrow = (V_high % 4 == 0) && aligned(logits, 16);
  q_stats_kernel<<<M, kStatThreads, 0, s>>>(logits, V_high, inv_tau, stats, vrow);
  vt_status st = launch_status("q_stats_kernel");
  if (st != VT_OK) return st;
  const int per_block = kFillThreads * kFillIds;
  dim3 grid((V + per_block - 1) / per_block, (M + kFillRows - 1) / kFillRows);
  q_fill_kernel<<<grid, kFillThreads, 0, s>>>(logits, M, V_high, f2t, V,
                                              inv_tau, stats, q, vec);
  return launch_status("q_fill_kernel");
}
