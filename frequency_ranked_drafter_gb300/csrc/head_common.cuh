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
// Workspace header shared by both head paths, so one workspace can serve
// calls of any M: bytes [0, 8) GEMV counters, [128, 132) tensor-core path
// error word, [1024, 2048) tensor-core per-row counters (M <= 256).  Every
// counter is zero between calls; nothing else is written in the header.
constexpr int kHeadTicketBytes = 2048;
constexpr int kHeadRowTicketOffset = 1024;
constexpr int kStageBytesMax = 96 * 1024;  // staged candidates, last CTA

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
  unsigned* ticket;      // [0]: CTAs done; [1]: next dynamically dealt row group
};

inline int head_pstride(int k) { return 2 + 2 * k; }

// Arrival on a grid-wide ticket: atomic increment with acquire-release
// semantics at gpu scope; returns the previous count.
__device__ __forceinline__ unsigned ticket_arrive(unsigned* ticket) {
  unsigned prev;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
               : "=r"(prev)
               : "l"(ticket)
               : "memory");
  return prev;
}

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

// Order-preserving image of a float in uint32 (larger float -> larger
// key; -0 and +0 share one key; -inf -> 0x007fffff, so 0 is below every
// real value).
__device__ __forceinline__ unsigned float_key(float f) {
  unsigned u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Shared-memory scratch of head_final_merge (8 warps).
struct MergeScratch {
  float w_val[8 * kTopKMax];  // level-1 winners of each warp
  int w_idx[8 * kTopKMax];
  float w_max[8];
  float w_sum[8];
};

// Merge of all CTAs' partial results, run by the last CTA of a launch
// (NT = 256 threads, 8 warps).  For every hidden state m:
//   Mg = max_b max_b;  Sg = sum_b sumexp_b * exp(max_b - Mg);
//   level 1: warp w merges lists [w*L, (w+1)*L) (L = ceil(G/8), at most
//            four lists per lane, their heads in registers) by a k-round
//            tournament; a round is a warp arg-max done with two redux.sync
//            (max of the order-preserving logit key, then min of the index
//            among the lanes holding it), after which the winning list
//            advances;
//   level 2: the 8*k level-1 winners are ranked by counting and the k best
//            written out by k threads at once (remap, exp, divide).
// All partials are read in one batch of independent loads (one L2 round
// trip) and the lists staged in shared memory (`stage`, G*k*8 bytes): this
// part runs on one SM while the others idle.  Its cost does not depend on
// the data.
template <int NT>
__device__ void head_final_merge(const HeadArgs& a, int MR, int G,
                                 float* stage, MergeScratch& sc) {
  static_assert(NT == 256, "merge layout assumes 8 warps");
  constexpr int kPer = kHeadMaxCtas / NT;      // CTA summaries per thread
  constexpr int kBatch = 16;                   // candidates per thread per batch
  constexpr int kOwn = kHeadMaxCtas / 8 / 32;  // lists per lane (level 1)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, ps = a.pstride, nc = G * k;
  float* sv = stage;
  int* si = reinterpret_cast<int*>(stage + nc);
  for (int m = 0; m < MR; ++m) {
    auto slot = [&](int b) { return a.part + ((size_t)b * MR + m) * ps; };
    float bm[kPer], bs[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = tid + j * NT;
      bm[j] = b < G ? __ldcg(slot(b)) : -INFINITY;
      bs[j] = b < G ? __ldcg(slot(b) + 1) : 0.f;
    }
    for (int base = 0; base < nc; base += NT * kBatch) {
      float cv[kBatch];
      int ci[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int c = base + j * NT + tid;
        if (c < nc) {
          const int b = c / k, r = c - b * k;
          cv[j] = __ldcg(slot(b) + 2 + r);
          ci[j] = __ldcg(reinterpret_cast<const int*>(slot(b)) + 2 + k + r);
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int c = base + j * NT + tid;
        if (c < nc) { sv[c] = cv[j]; si[c] = ci[j]; }
      }
    }
    float wm = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPer; ++j) wm = fmaxf(wm, bm[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(~0u, wm, o));
    if (lane == 0) sc.w_max[warp] = wm;
    __syncthreads();  // publishes the stage and the warp maxima
    float mg = sc.w_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) mg = fmaxf(mg, sc.w_max[w]);
    float ws = 0.f;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (bs[j] > 0.f) ws += bs[j] * __expf(bm[j] - mg);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(~0u, ws, o);
    if (lane == 0) sc.w_sum[warp] = ws;

    // ---- level 1: per-warp tournament over its lists
    {
      const int L = (G + 7) / 8;
      const int b0 = warp * L, b1 = min(G, b0 + L);
      int hd[kOwn];
      float hv[kOwn];
      int hi[kOwn];
#pragma unroll
      for (int o = 0; o < kOwn; ++o) {
        const int b = b0 + lane + 32 * o;
        hd[o] = 0;
        hv[o] = b < b1 ? sv[b * k] : -INFINITY;
        hi[o] = b < b1 ? si[b * k] : INT_MAX;
      }
      float rv = -INFINITY;
      int ri = INT_MAX;
      for (int r = 0; r < k; ++r) {
        float lv = -INFINITY;
        int li = INT_MAX, lo = 0;
#pragma unroll
        for (int o = 0; o < kOwn; ++o)
          if (hi[o] != INT_MAX && key_beats(hv[o], hi[o], lv, li)) {
            lv = hv[o]; li = hi[o]; lo = o;
          }
        const unsigned lk = li != INT_MAX ? float_key(lv) : 0u;
        const unsigned wk = __reduce_max_sync(~0u, lk);
        if (wk == 0u) break;  // this warp's lists are exhausted
        const int wi = (int)__reduce_min_sync(
            ~0u, lk == wk ? (unsigned)li : 0xffffffffu);
        const unsigned owner = __ballot_sync(~0u, lk == wk && li == wi);
        const int ol = __ffs(owner) - 1;
        const float wv = __shfl_sync(~0u, lv, ol);
        if (lane == r) { rv = wv; ri = wi; }
        if (lane == ol) {  // the winning list advances
#pragma unroll
          for (int o = 0; o < kOwn; ++o)
            if (o == lo) {
              const int b = b0 + lane + 32 * o;
              const int h = ++hd[o];
              hv[o] = h < k ? sv[b * k + h] : -INFINITY;
              hi[o] = h < k ? si[b * k + h] : INT_MAX;
            }
        }
      }
      if (lane < k) { sc.w_val[warp * k + lane] = rv; sc.w_idx[warp * k + lane] = ri; }
    }
    __syncthreads();

    // ---- level 2: rank the 8*k level-1 winners, write the k best
    float sg = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sg += sc.w_sum[w];
    int32_t* ids = a.out_ids + (size_t)m * k;
    float* probs = a.out_probs + (size_t)m * k;
    for (int c = tid; c < 8 * k; c += NT) {
      const float v = sc.w_val[c];
      const int i = sc.w_idx[c];
      if (i == INT_MAX) continue;
      int rank = 0;
      for (int q = 0; q < 8 * k; ++q)
        rank += key_beats(sc.w_val[q], sc.w_idx[q], v, i);
      if (rank < k) {
        ids[rank] = a.t2f ? a.t2f[i] : i;
        probs[rank] = expf(v - mg) / sg;
      }
    }
    __syncthreads();
  }
}

// CUDA-core GEMV path (M = 1 in vt_draft_head; up to 4 per launch), head_gemv.cu.
vt_status head_gemv(const HeadArgs& a, const DeviceInfo& di, cudaStream_t s);

// Tree-draft tensor-core path (M >= kHeadTcMinM), head_tc.cu.  The
// workspace holds an error word at byte 128, per-row counters and partials
// and, when out_logits is null, the [M, V_high] fp32 logits.
constexpr int kHeadTcMinM = 2;
size_t head_tc_workspace(int M, int V_high, int k);
vt_status head_tc(const uint16_t* H, int M, int d, int64_t ldh,
                  const uint16_t* W, int V_high, const int32_t* t2f, int k,
                  int32_t* out_ids, float* out_probs, float* out_logits,
                  void* ws, const DeviceInfo& di, cudaStream_t s);

}  // namespace vt
