// Pieces shared by the two vt_draft_head paths (CUDA-core GEMV for small M,
// tensor-core skinny GEMM for tree drafts): the argument block, the
// workspace layout, and the cross-CTA merge run by the last CTA.
#pragma once

#include <float.h>
#include <limits.h>

#include "tc_ptx.cuh"
#include "vt_checks.cuh"
#include "vt_common.cuh"

namespace vt {

constexpr int kTopKMax = 32;
constexpr int kHeadMaxCtas = 1024;
// Workspace header shared by both head paths, so one workspace can serve
// calls of any M: bytes [0, 8) GEMV counters, [128, 132) device error word
// (both paths), [1024, 2048) tensor-core per-row counters (M <= 256).  Every
// counter is zero between calls; nothing else is written in the header.
constexpr int kHeadTicketBytes = 2048;
constexpr int kHeadRowTicketOffset = 1024;
constexpr int kStageBytesMax = 96 * 1024;  // staged candidates, last CTA

// Options of a head call (vt_head_options): kept-row bias added to every
// logit, temperature T (probabilities are softmax(logit / T); the kernels
// multiply by the fp32 reciprocal of T, exact for T = 1), and the
// selection: the k largest logit / T, or (sample) the k largest
// logit / T + g with g the Gumbel noise of the token (gumbel_noise).
struct HeadOpts {
  const float* bias;  // [V_high] or null
  float tau;
  int sample;
  uint64_t seed, offset;
  const int32_t* row_ids = nullptr;  // device; the noise index of each hidden
                                     // state of the launch (null: its row)
};

// Each CTA b publishes, per hidden state m, one record of `pstride` 32-bit
// words at part + (m * G + b) * pstride (G CTAs), 16-byte aligned so that
// the records of one m are a single bulk copy:
//   [0] max of logit/T over its rows, [1] sum of exp(logit/T - max),
//   [2, 4) unused, [4, 4+2k) its k best entries as 64-bit keys of
//   (selection score, full-vocabulary id) (make_key), best first, unused
//   slots kEmptyKey; sampling only: [4+2k, 4+3k) the entries' logit/T.
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
  float* part;         // [M][grid][pstride]
  int pstride;
  unsigned* ticket;      // [0]: CTAs done; [1]: next dynamically dealt row group
  unsigned* err;         // device error word (VT_ERR_TIMEOUT if a wait gave up)
  HeadOpts opt;
  int m_base;            // index of this launch's first hidden state in the call
};

inline int head_pstride(int k, bool sample) {
  return (4 + (sample ? 3 : 2) * k + 3) / 4 * 4;
}

// Workspace of one GEMV launch over MR hidden states: the shared header and
// up to kHeadMaxCtas CTAs' partials.
inline size_t head_gemv_workspace(int MR, int k, bool sample) {
  return (size_t)kHeadTicketBytes +
         (size_t)kHeadMaxCtas * MR * head_pstride(k, sample) * sizeof(float);
}

// Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and
// Shaw ("Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011): ten rounds,
// each multiplying counter words 0 and 2 by the round multipliers (high and
// low halves of the 64-bit products) and mixing in the key, which advances by
// the Weyl increments between rounds.  Returns output word 0.
__device__ __forceinline__ uint32_t philox4x32_10_w0(uint32_t c0, uint32_t c1,
                                                     uint32_t c2, uint32_t c3,
                                                     uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

// Gumbel noise of token `full_id` for hidden state m at step (seed, offset):
// x = word 0 of Philox4x32-10 at counter (full_id, m, offset low, offset
// high), key (seed low, seed high); u = ((x >> 9) + 1/2) / 2^23 in (0, 1),
// exact in binary32; g = -log(-log(u)).  Keyed by the full-vocabulary id, so
// a token's noise does not depend on which tokens were kept or where.
__device__ __forceinline__ float gumbel_noise(uint64_t seed, uint64_t offset,
                                              int m, int full_id) {
  const uint32_t x = philox4x32_10_w0((uint32_t)full_id, (uint32_t)m,
                                      (uint32_t)offset, (uint32_t)(offset >> 32),
                                      (uint32_t)seed, (uint32_t)(seed >> 32));
  const float u = ((float)(x >> 9) + 0.5f) * 0x1p-23f;
  return -logf(-logf(u));
}

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

// Order-preserving image of a float in uint32 (larger float -> larger
// key; -0 and +0 share one key; -inf -> 0x007fffff, so 0 is below every
// real value).
__device__ __forceinline__ unsigned float_key(float f) {
  unsigned u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of float_key (-0 comes back as +0).
__device__ __forceinline__ float key_float(unsigned u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// One 64-bit key per (logit, id) entry: larger logit first, then lower id
// (the GEMV path keys full-vocabulary ids, so its ties fall exactly as the
// oracle's).  Distinct ids give distinct keys; an empty slot (-inf,
// INT_MAX) is kEmptyKey, below every real entry.
typedef unsigned long long entry_key;
__device__ __forceinline__ entry_key make_key(float v, int i) {
  return ((entry_key)float_key(v) << 32) | (unsigned)~i;
}
__device__ __forceinline__ float key_logit(entry_key x) {
  return key_float((unsigned)(x >> 32));
}
__device__ __forceinline__ int key_id(entry_key x) { return ~(int)(unsigned)x; }
constexpr entry_key kEmptyKey = 0x007fffff80000000ull;

// Double-buffered hand-over slots of cta_merge_lists for W <= 16 warps.
constexpr int kMergeMaxWarps = 16;
struct ListSlots {
  entry_key key[2][kMergeMaxWarps / 2][32];
  int val[2][kMergeMaxWarps / 2][32];
};

// Merges the sorted 32-entry lists (best first, lane j holds the j-th) that
// the W warps of the CTA hold in (x, y) into warp 0, which ends with the 32
// best of all of them, sorted.  Per level, the upper half of the remaining
// warps hands its lists over through shared memory; each lower warp takes
// max(own[j], other[31 - j]) -- the 32 best of both as a bitonic sequence --
// and sorts it with five compare-exchange stages.  One barrier per level;
// `level` counts levels across calls so the slots alternate.  Every thread
// of the CTA must call it.
template <int W, bool kPayload>
__device__ __forceinline__ void cta_merge_lists(entry_key& x, int& y, ListSlots& ls,
                                                int& level) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int half = W / 2; half >= 1; half >>= 1, ++level) {
    const int buf = level & 1;
    if (warp >= half && warp < 2 * half) {
      ls.key[buf][warp - half][lane] = x;
      if (kPayload) ls.val[buf][warp - half][lane] = y;
    }
    __syncthreads();
    if (warp < half) {
      const entry_key ox = ls.key[buf][warp][31 - lane];
      if (ox > x) {
        x = ox;
        if (kPayload) y = ls.val[buf][warp][31 - lane];
      }
#pragma unroll
      for (int st = 16; st > 0; st >>= 1) {
        const entry_key px = __shfl_xor_sync(~0u, x, st);
        const int py = kPayload ? __shfl_xor_sync(~0u, y, st) : 0;
        if (((lane & st) == 0) ? (px > x) : (x > px)) {
          x = px;
          if (kPayload) y = py;
        }
      }
    }
  }
}

// Shared-memory scratch of head_final_merge.
struct MergeScratch {
  ListSlots slots;
  entry_key surv[kTopKMax * kTopKMax];  // entries reaching the k-th head
  float surv_s[kTopKMax * kTopKMax];    // ... their logit/T (sampling)
  int q_list[kTopKMax];                 // the lists with the k best heads
  float w_max[kMergeMaxWarps];
  float w_sum[kMergeMaxWarps];
  entry_key t_key;                      // the k-th best head
  int cnt;
};

// Bitonic sort, descending, of the 32*E keys a warp holds E per lane
// (element i = lane + 32*r sits in register r); y rides along with its key.
template <int E>
__device__ __forceinline__ void warp_bitonic_desc(entry_key (&x)[E], int (&y)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32 * E; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int r = 0; r < E; ++r) {
        const int i = lane + 32 * r;
        // the lower element of a pair keeps the larger key in descending runs
        const bool desc = (i & size) == 0;
        if (stride >= 32) {  // partner in another register of this lane
          const int rp = r ^ (stride >> 5);
          if (r < rp && desc != (x[r] > x[rp])) {
            const entry_key tx = x[r]; x[r] = x[rp]; x[rp] = tx;
            const int ty = y[r]; y[r] = y[rp]; y[rp] = ty;
          }
        } else {
          const entry_key px = __shfl_xor_sync(~0u, x[r], stride);
          const int py = __shfl_xor_sync(~0u, y[r], stride);
          const bool lower = (i & stride) == 0;
          if ((desc == lower) != (x[r] > px)) {
            x[r] = px;
            y[r] = py;
          }
        }
      }
    }
  }
}

// The 32 best list heads (list(b)[0]) of one warp's share b0 .. b1-1,
// sorted, one per lane, with their list numbers; empty slots are
// (kEmptyKey, -1).
template <int E, class List>
__device__ __forceinline__ void warp_top_heads(const List& list, int b0, int b1,
                                               entry_key& ox, int& oy) {
  const int lane = threadIdx.x & 31;
  entry_key x[E];
  int y[E];
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const int b = b0 + lane + 32 * r;
    x[r] = b < b1 ? list(b)[0] : kEmptyKey;
    y[r] = b < b1 ? b : -1;
  }
  warp_bitonic_desc<E>(x, y);
  ox = x[0];
  oy = y[0];
}

// Same for 32 < b1 - b0 <= 64 heads, of which only the k best need to be
// exact: the first 32 are sorted in registers, then the others that beat
// the list's k-th key (ballot; few) are inserted one at a time, the last lane
// dropping out.  The list stays sorted and holds only real heads, and its
// first k entries are the share's k best: enough for cta_merge_lists to
// give the k best of all.
template <class List>
__device__ __forceinline__ void warp_top_heads_ins(const List& list, int b0, int b1,
                                                   int k, entry_key& ox, int& oy) {
  const int lane = threadIdx.x & 31;
  entry_key x[1];
  int y[1];
  {
    const int b = b0 + lane;
    x[0] = b < b1 ? list(b)[0] : kEmptyKey;
    y[0] = b < b1 ? b : -1;
  }
  const int b = b0 + 32 + lane;
  const entry_key x1 = b < b1 ? list(b)[0] : kEmptyKey;  // loaded before the sort
  warp_bitonic_desc<1>(x, y);
  entry_key thr = __shfl_sync(~0u, x[0], k - 1);
  unsigned cand = __ballot_sync(~0u, x1 > thr);
  while (cand) {  // warp-uniform
    const int src = __ffs(cand) - 1;
    const entry_key ck = __shfl_sync(~0u, x1, src);
    const int p = __popc(__ballot_sync(~0u, x[0] > ck));
    const entry_key up = __shfl_up_sync(~0u, x[0], 1);
    const int upy = __shfl_up_sync(~0u, y[0], 1);
    if (lane == p) {
      x[0] = ck;
      y[0] = b0 + 32 + src;
    } else if (lane > p) {
      x[0] = up;
      y[0] = upy;
    }
    thr = __shfl_sync(~0u, x[0], k - 1);
    cand &= ~(1u << src);
    cand &= __ballot_sync(~0u, x1 > thr);
  }
  ox = x[0];
  oy = y[0];
}

// Merge of all CTAs' partial results, run by the last CTA of a launch
// (NT threads, W = NT/32 warps).  Each CTA published (max, sumexp) and its
// k best entries as sorted keys, so for every hidden state m:
//   Mg = max_b max_b;  Sg = sum_b sumexp_b * exp(max_b - Mg);
//   the top-k lies in the k lists whose heads are best (a list whose head
//   is beaten by k other heads holds nothing that k entries do not beat),
//   and within them in the entries at least as good as T, the k-th best
//   head: at most k*k survivors.  Each warp bitonic-sorts the heads of its
//   share of the lists in registers, the warps' sorted heads are merged in
//   registers (cta_merge_lists) to give the k best lists and T, and the
//   survivors are ranked by counting; the k best write their id and
//   exp(l - Mg) / Sg.
// The G records of one m are contiguous and reach shared memory (`stage`,
// G * pstride words, 16-byte aligned) in one bulk copy -- one L2 round trip
// without a load per entry; this part runs on one SM while the others idle.
// The work does not depend on the data.  If the copy does not land within
// the wait budget the error word is set and the merge gives up.
template <int NT>
__device__ void head_final_merge(const HeadArgs& a, int MR, int G, float* stage,
                                 MergeScratch& sc, uint64_t* bar) {
  constexpr int W = NT / 32;
  static_assert(W >= 8 && W <= kMergeMaxWarps, "merge layout: 8 to 16 warps");
  constexpr int kPer = kHeadMaxCtas / NT;  // CTA records per thread
  constexpr int kSortE = kHeadMaxCtas / W / 32;  // heads per lane, <= 4
  constexpr long long kWaitBudget = 1ll << 31;   // SM cycles, about a second
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, ps = a.pstride;
  const uint32_t bytes = (uint32_t)G * ps * sizeof(float);
  int level = 0;
  auto list = [&](int b) {
    return reinterpret_cast<const entry_key*>(stage + (size_t)b * ps + 4);
  };
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  for (int m = 0; m < MR; ++m) {
    if (tid == 0) {
      // the other CTAs' records were acquired through the ticket (generic
      // proxy); earlier generic use of `stage` is done (barrier above)
      asm volatile("fence.proxy.async.global;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc::mbar_arrive_expect_tx(bar, bytes);
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
          " [%0], [%1], %2, [%3];" ::"r"(tc::smem_u32(stage)),
          "l"(a.part + (size_t)m * G * ps), "r"(bytes), "r"(tc::smem_u32(bar))
          : "memory");
      sc.cnt = 0;
    }
    if (!tc::mbar_wait(bar, m & 1, kWaitBudget)) {
      if (tid == 0) atomicExch(a.err, (unsigned)VT_ERR_TIMEOUT);
      tc::mbar_wait(bar, m & 1, kWaitBudget);  // let the copy finish
      return;
    }
    float2 st[kPer];  // this thread's CTA records' (max, sumexp)
    float lm = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = tid + j * NT;
      st[j] = b < G ? *reinterpret_cast<const float2*>(stage + (size_t)b * ps)
                    : make_float2(-INFINITY, 0.f);
      lm = fmaxf(lm, st[j].x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lm = fmaxf(lm, __shfl_xor_sync(~0u, lm, o));
    if (lane == 0) sc.w_max[warp] = lm;
    entry_key hx;
    int hy;
    {
      const int L = (G + W - 1) / W;
      const int b0 = warp * L, b1 = min(G, b0 + L);
      if (L <= 32) warp_top_heads<1>(list, b0, b1, hx, hy);
      else if (L <= 64) warp_top_heads_ins(list, b0, b1, k, hx, hy);
      else warp_top_heads<kSortE>(list, b0, b1, hx, hy);
    }
    // the k best heads of all, in order (distinct: lists hold disjoint ids);
    // the first barrier inside also publishes the warp maxima
    cta_merge_lists<W, true>(hx, hy, sc.slots, level);
    if (warp == 0 && lane < k) {
      sc.q_list[lane] = hy;
      if (lane == k - 1) sc.t_key = hx;
    }
    __syncthreads();
    const entry_key t = sc.t_key;
    for (int c = tid; c < k * k; c += NT) {
      const int j = c / k;
      const int b = sc.q_list[j];
      if (b < 0) continue;
      const entry_key x = list(b)[c - j * k];
      if (x >= t && x != kEmptyKey) {
        const int p = atomicAdd(&sc.cnt, 1);
        sc.surv[p] = x;
        if (a.opt.sample)
          sc.surv_s[p] = reinterpret_cast<const float*>(list(b) + k)[c - j * k];
      }
    }
    float mg = sc.w_max[0];
#pragma unroll
    for (int w = 1; w < W; ++w) mg = fmaxf(mg, sc.w_max[w]);
    float ws = 0.f;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (st[j].y > 0.f) ws += st[j].y * __expf(st[j].x - mg);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(~0u, ws, o);
    if (lane == 0) sc.w_sum[warp] = ws;
    __syncthreads();
    float sg = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) sg += sc.w_sum[w];
    const int S = sc.cnt;
    int32_t* ids = a.out_ids + (size_t)m * k;
    float* probs = a.out_probs + (size_t)m * k;
    // (sampling: the key is the score; the logit/T of list entries follows
    // the keys in the record)
    for (int c = tid; c < S; c += NT) {
      const entry_key x = sc.surv[c];
      int rank = 0;
      for (int q = 0; q < S; ++q) rank += sc.surv[q] > x;
      if (rank < k && VT_CHECKED(m < MR)) {
        ids[rank] = key_id(x);
        const float sv = a.opt.sample ? sc.surv_s[c] : key_logit(x);
        probs[rank] = expf(sv - mg) / sg;
      }
    }
    __syncthreads();
  }
}

// CUDA-core GEMV path (M = 1 in vt_draft_head; up to 4 per launch), head_gemv.cu.
vt_status head_gemv(const HeadArgs& a, const DeviceInfo& di, cudaStream_t s);

// vt_draft_head_ex with a device map giving each hidden state's noise index
// (its row in the caller's batch); the sets entry point uses it (head_api.cu).
vt_status draft_head_rows(const uint16_t* H, int32_t M, int32_t d, int64_t ldh,
                          const uint16_t* W_high, int32_t V_high,
                          const int32_t* t2f, int32_t k,
                          const vt_head_options* opts, const int32_t* row_ids,
                          int32_t* out_ids, float* out_probs, void* ws,
                          size_t ws_bytes, void* stream);

// Tree-draft tensor-core path (M >= kHeadTcMinM), head_tc.cu.  The
// workspace holds an error word at byte 128, per-row counters and partials
// and, when out_logits is null, the [M, V_high] fp32 logits.
constexpr int kHeadTcMinM = 2;
size_t head_tc_workspace(int M, int V_high, int k);
vt_status head_tc(const uint16_t* H, int M, int d, int64_t ldh,
                  const uint16_t* W, int V_high, const int32_t* t2f, int k,
                  const HeadOpts& opt, int32_t* out_ids, float* out_probs,
                  float* out_logits, void* ws, const DeviceInfo& di,
                  cudaStream_t s);

}  // namespace vt
