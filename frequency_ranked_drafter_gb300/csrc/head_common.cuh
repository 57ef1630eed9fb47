// Pieces shared by the two vt_draft_head paths (CUDA-core GEMV for small M,
// tensor-core skinny GEMM for tree drafts): the argument block, the
// workspace layout, and the cross-CTA merge run by the last CTA.
#pragma once

#include <float.h>
#include <limits.h>

#include "vt_common.cuh"

namespace vt {

constexpr int kTopKMax = 32;
constexpr int kHeadMaxCtas = 1024;
constexpr int kHeadTicketBytes = 256;
constexpr int kSurvivorCap = 1024;
constexpr int kStageBytesMax = 160 * 1024;  // staged partials, last CTA

// Each CTA publishes, per hidden state m, `pstride` 32-bit words:
//   [0] max logit of its rows, [1] sum of exp(logit - max) over its rows,
//   [2, 2+k) its k best logits (descending), [2+k, 2+2k) their trimmed
//   indices (int bits); unused slots hold (-inf, INT_MAX).
struct HeadArgs {
  const uint16_t* H;
  int64_t ldh;
  int M;  // hidden states handled by this launch
  int d;
  const uint16_t* W;
  int V_high;
  const int32_t* t2f;
  int k;
  int32_t* out_ids;    // [M, k]
  float* out_probs;    // [M, k]
  float* out_logits;   // [M, V_high] or null
  float* part;         // [grid][M][pstride]
  int pstride;
  unsigned* ticket;
};

inline int head_pstride(int k) { return 2 + 2 * k; }

__device__ __forceinline__ bool key_beats(float v, int i, float v2, int i2) {
  return v > v2 || (v == v2 && i < i2);
}

// Block-wide reductions for NT threads; scratch holds NT/32 entries.
template <int NT>
__device__ __forceinline__ float block_max(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(~0u, v, o));
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = scratch[0];
  for (int w = 1; w < NT / 32; ++w) r = fmaxf(r, scratch[w]);
  __syncthreads();
  return r;
}

template <int NT>
__device__ __forceinline__ float block_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < NT / 32; ++w) r += scratch[w];
  __syncthreads();
  return r;
}

template <int NT>
__device__ __forceinline__ void block_best(float& v, int& i, float* sv,
                                          int* si) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(~0u, v, o);
    const int i2 = __shfl_xor_sync(~0u, i, o);
    if (key_beats(v2, i2, v, i)) { v = v2; i = i2; }
  }
  if ((threadIdx.x & 31) == 0) { sv[threadIdx.x >> 5] = v; si[threadIdx.x >> 5] = i; }
  __syncthreads();
  v = sv[0];
  i = si[0];
  for (int w = 1; w < NT / 32; ++w)
    if (key_beats(sv[w], si[w], v, i)) { v = sv[w]; i = si[w]; }
  __syncthreads();
}

// Merge of all CTAs' partial results, run by the last CTA of a launch.
// `stage` is shared memory of at least G * pstride words (the caller sizes
// the launch so that it fits).  For every hidden state m:
//   global max  Mg = max_b max_b;   Sg = sum_b sumexp_b * exp(max_b - Mg);
//   threshold   T0 = the best of the CTAs' k-th entries: the global k-th
//               entry can be no worse, so only entries not beaten by T0 can
//               be in the global top-k (usually about k of them);
//   ranks       of those survivors by counting, written out in order.
// If more than kSurvivorCap entries survive (adversarial inputs), the top-k
// falls back to k rounds of a block-wide arg-max.
template <int NT>
__device__ void head_final_merge(const HeadArgs& a, int MR, int G,
                                 float* stage, float* red_v, int* red_i,
                                 float2* surv, int* s_cnt) {
  const int tid = threadIdx.x;
  const int k = a.k, ps = a.pstride;
  int* stage_i = reinterpret_cast<int*>(stage);
  for (int m = 0; m < MR; ++m) {
    for (int t = tid; t < G * ps; t += NT) {
      const int b = t / ps, o = t % ps;
      stage[t] = __ldcg(a.part + ((size_t)b * MR + m) * ps + o);
    }
    if (tid == 0) *s_cnt = 0;
    __syncthreads();

    float mg = -INFINITY, t0v = -INFINITY;
    int t0i = INT_MAX;
    for (int b = tid; b < G; b += NT) {
      mg = fmaxf(mg, stage[b * ps]);
      const float kv = stage[b * ps + 2 + k - 1];
      const int ki = stage_i[b * ps + 2 + 2 * k - 1];
      if (key_beats(kv, ki, t0v, t0i)) { t0v = kv; t0i = ki; }
    }
    mg = block_max<NT>(mg, red_v);
    block_best<NT>(t0v, t0i, red_v, red_i);
    float sg = 0.f;
    for (int b = tid; b < G; b += NT) {
      const float s = stage[b * ps + 1];
      if (s > 0.f) sg += s * __expf(stage[b * ps] - mg);
    }
    sg = block_sum<NT>(sg, red_v);

    for (int c = tid; c < G * k; c += NT) {
      const int b = c / k, j = c % k;
      const float v = stage[b * ps + 2 + j];
      const int i = stage_i[b * ps + 2 + k + j];
      if (i != INT_MAX && !key_beats(t0v, t0i, v, i)) {
        const int p = atomicAdd(s_cnt, 1);
        if (p < kSurvivorCap) surv[p] = make_float2(v, __int_as_float(i));
      }
    }
    __syncthreads();
    const int S = *s_cnt;
    int32_t* ids = a.out_ids + (size_t)m * k;
    float* probs = a.out_probs + (size_t)m * k;
    if (S <= kSurvivorCap) {
      for (int s = tid; s < S; s += NT) {
        const float v = surv[s].x;
        const int i = __float_as_int(surv[s].y);
        int rank = 0;
        for (int q = 0; q < S; ++q)
          rank += key_beats(surv[q].x, __float_as_int(surv[q].y), v, i);
        if (rank < k) {
          ids[rank] = a.t2f ? a.t2f[i] : i;
          probs[rank] = expf(v - mg) / sg;
        }
      }
    } else {
      float pv = INFINITY;
      int pi = INT_MIN;
      for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int c = tid; c < G * k; c += NT) {
          const int b = c / k, j = c % k;
          const float v = stage[b * ps + 2 + j];
          const int i = stage_i[b * ps + 2 + k + j];
          if (i != INT_MAX && key_beats(pv, pi, v, i) &&
              key_beats(v, i, bv, bi)) { bv = v; bi = i; }
        }
        block_best<NT>(bv, bi, red_v, red_i);
        if (tid == 0) {
          const bool ok = bi != INT_MAX;
          ids[r] = !ok ? -1 : (a.t2f ? a.t2f[bi] : bi);
          probs[r] = ok ? expf(bv - mg) / sg : 0.f;
        }
        pv = bv;
        pi = bi;
      }
    }
    __syncthreads();
  }
}

// Small-M GEMV path (M <= 4), head_gemv.cu.
vt_status head_gemv(const HeadArgs& a, const DeviceInfo& di, cudaStream_t s);

}  // namespace vt
