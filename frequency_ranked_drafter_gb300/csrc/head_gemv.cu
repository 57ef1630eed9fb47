// vt_draft_head, small-M path: split-V GEMV fused with the softmax over the
// kept rows, top-k and the trimmed -> full remap.
//
// "FR-Spec: Accelerating Large-Vocabulary Language Models via
// Frequency-Ranked Speculative Sampling", Method > Key design: the draft
// lm_head projects onto the V_high most frequent tokens only and the softmax
// is computed on that subset.  "VocabTrim: ...", Implementation Step 4:
// softmax of the drafter logits, then trimmed index -> full id through
// trimmed_to_full.
//
// At one hidden state the head is a GEMV bound by reading W_high once
// (V_high * d * 2 bytes).  One launch does everything:
//   * one CTA of 16 warps per SM; every warp streams groups of rows of
//     W_high (two rows at d > 1024, 8 chunks of 16 bytes per lane of each
//     in flight) and dots them with H, which each CTA keeps in shared memory
//     as fp32; most groups are dealt round-robin over all warps of the grid
//     and the last eighth one at a time from a counter, so every SM streams
//     about the same bytes and all finish together;
//   * launched as a programmatic dependent of the kernel ahead of it: the
//     grid becomes resident while that kernel finishes and prefetches its
//     first rows into L2, reading nothing that kernel may write until it
//     has ended (griddepcontrol.wait);
//   * each warp keeps, per hidden state, an online (max, sum of exp) of
//     s = (logit + bias) / T and a sorted list of its k best entries, one
//     64-bit key of (score, full id) per lane (insertion by ballot and a
//     one-lane shift), so no logit is ever written to memory; the score is s
//     for top-k and s + Gumbel noise of the token when sampling ("VocabTrim",
//     Step 4 draws from the trimmed softmax; the Gumbel-max rule draws from
//     the same distribution);
//   * each CTA merges its warps' lists in registers (cta_merge_lists) and
//     publishes (max, sumexp, top-k) to the workspace; the last CTA to finish
//     (atomic ticket, no waiting) merges all CTAs (head_final_merge),
//     rescales the sums, writes ids and probabilities and re-arms the ticket.
#include <float.h>

#include "head_common.cuh"

namespace vt {
namespace {

// One CTA of 16 warps per SM: half the records of two 8-warp CTAs for the
// last CTA to merge, the same loads in flight.
constexpr int kGemvThreads = 512;
constexpr int kGemvWarps = kGemvThreads / 32;
// Row groups per warp prefetched into L2 before the dependency wait.
constexpr int kGemvPrefetchGroups = 2;

__device__ __forceinline__ float dot8(uint4 w, float4 h0, float4 h1,
                                      float acc) {
  acc = fmaf(bf16lo(w.x), h0.x, acc);
  acc = fmaf(bf16hi(w.x), h0.y, acc);
  acc = fmaf(bf16lo(w.y), h0.z, acc);
  acc = fmaf(bf16hi(w.y), h0.w, acc);
  acc = fmaf(bf16lo(w.z), h1.x, acc);
  acc = fmaf(bf16hi(w.z), h1.y, acc);
  acc = fmaf(bf16lo(w.w), h1.z, acc);
  acc = fmaf(bf16hi(w.w), h1.w, acc);
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  return v;
}

template <int MR, int CPL, int U, bool kSample>
__global__ void __launch_bounds__(kGemvThreads, 1)
    head_gemv_kernel(HeadArgs a) {
  extern __shared__ __align__(16) float hs[];  // [MR][d] fp32 hidden states
  __shared__ float w_mx[MR][kGemvWarps], w_se[MR][kGemvWarps];
  __shared__ MergeScratch msc;
  __shared__ uint64_t merge_bar;
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = a.d, k = a.k;

  const int nchunks = d >> 3;
  const int nkb = (nchunks + 32 * CPL - 1) / (32 * CPL);
  const int gwarps = gridDim.x * kGemvWarps;
  const int gwarp = blockIdx.x * kGemvWarps + warp;
  const int ngroups = (a.V_high + U - 1) / U;
  const int static_rounds = (ngroups / gwarps) * 7 / 8;

  // Launched as a programmatic dependent: this grid can be resident while
  // the kernel ahead of it (the previous draft step's merge, or the layer
  // that wrote H) finishes.  Meanwhile each warp only asks L2 for the first
  // row groups it will stream (weights; a prefetch is a hint, the loads that
  // use them follow the wait), then waits before reading H, t2f, the bias
  // or the workspace.
  grid_launch_dependents();
  if (lane < min(kGemvPrefetchGroups, static_rounds)) {
    const int r0 = (gwarp + lane * gwarps) * U;
    const int nr = min(U, a.V_high - r0);
    prefetch_l2(a.W + (int64_t)r0 * d, (uint32_t)(nr * d * 2));
  }
  grid_dependency_wait();

  // H (bf16, row stride ldh) -> fp32 shared memory, two values per word.
  for (int m = 0; m < MR; ++m) {
    const uint32_t* src =
        reinterpret_cast<const uint32_t*>(a.H + (int64_t)m * a.ldh);
    float2* dst = reinterpret_cast<float2*>(hs + m * d);
    for (int j = tid; j < d / 2; j += kGemvThreads) {
      const uint32_t x = src[j];
      dst[j] = make_float2(bf16lo(x), bf16hi(x));
    }
  }
  __syncthreads();

  // Per hidden state: running max and sum of exp of s = logit / T (online
  // softmax), and the warp's k best entries as keys of (score, full id),
  // lane j holding the j-th best, with thr the k-th.  The score is s, or
  // s + Gumbel noise when sampling; then ts carries each entry's s.
  float mx[MR], se[MR], ts[MR];
  entry_key tk[MR], thr[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    mx[m] = -INFINITY; se[m] = 0.f; ts[m] = -INFINITY;
    tk[m] = kEmptyKey; thr[m] = kEmptyKey;
  }
  const float* bias = a.opt.bias;
  int mrow[MR];  // noise index of each hidden state
#pragma unroll
  for (int m = 0; m < MR; ++m)
    mrow[m] = a.opt.row_ids ? __ldg(a.opt.row_ids + a.m_base + m) : a.m_base + m;
  const float inv_tau = 1.0f / a.opt.tau;

  const float4* h4 = reinterpret_cast<const float4*>(hs);

  auto process_group = [&](int g) {
    const int r0 = g * U;
    // full ids (and biases) of the group's rows, fetched while the rows
    // stream in
    int fid[U];
    float brow[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = min(r0 + u, a.V_high - 1);
      fid[u] = a.t2f ? __ldg(a.t2f + row) : row;
      brow[u] = bias ? __ldg(bias + row) : 0.f;
    }
    float noise[U][MR];
    float acc[U][MR];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int m = 0; m < MR; ++m) acc[u][m] = 0.f;

    for (int kb = 0; kb < nkb; ++kb) {
      uint4 wv[U][CPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int row = min(r0 + u, a.V_high - 1);  // clamp: tail rows unused
        const uint4* wrow =
            reinterpret_cast<const uint4*>(a.W + (int64_t)row * d);
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          const int c = kb * 32 * CPL + lane + 32 * j;
          wv[u][j] = c < nchunks ? ld_stream_u4(wrow + c) : make_uint4(0, 0, 0, 0);
        }
      }
      if (kSample && kb == 0) {  // generator work overlaps the row loads
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int m = 0; m < MR; ++m)
            noise[u][m] = gumbel_noise(a.opt.seed, a.opt.offset, mrow[m], fid[u]);
      }
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = kb * 32 * CPL + lane + 32 * j;
        if (c < nchunks) {
#pragma unroll
          for (int m = 0; m < MR; ++m) {
            const float4 h0 = h4[(m * d >> 2) + 2 * c];
            const float4 h1 = h4[(m * d >> 2) + 2 * c + 1];
#pragma unroll
            for (int u = 0; u < U; ++u) acc[u][m] = dot8(wv[u][j], h0, h1, acc[u][m]);
          }
        }
      }
    }

#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = r0 + u;
      if (row >= a.V_high) break;
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        const float l = warp_sum(acc[u][m]) + brow[u];
        if (a.out_logits && lane == 0)
          a.out_logits[(int64_t)m * a.V_high + row] = l;
        const float sv = l * inv_tau;  // exact for T = 1
        if (sv > mx[m]) {
          se[m] = se[m] * __expf(mx[m] - sv) + 1.f;
          mx[m] = sv;
        } else {
          se[m] += __expf(sv - mx[m]);
        }
        const entry_key key = make_key(kSample ? sv + noise[u][m] : sv, fid[u]);
        if (key > thr[m]) {  // insert at its rank, the k-th drops out
          const int p = __popc(__ballot_sync(~0u, lane < k && tk[m] > key));
          const entry_key up = __shfl_up_sync(~0u, tk[m], 1);
          const float ups = kSample ? __shfl_up_sync(~0u, ts[m], 1) : 0.f;
          if (lane == p) {
            tk[m] = key;
            ts[m] = sv;
          } else if (lane > p && lane < k) {
            tk[m] = up;
            ts[m] = ups;
          }
          thr[m] = __shfl_sync(~0u, tk[m], k - 1);
        }
      }
    }
  };

  // Rows are dealt in groups of U.  Most groups go round-robin over all
  // warps of the grid; the last ~1/8 are handed out one at a time from a
  // global counter, so warps that stream faster take more and all warps
  // finish together.  A warp asks for its next dynamic group one group ahead.
  const int n_static = static_rounds * gwarps;
  int g_next = 0;
  if (lane == 0) g_next = (int)atomicAdd(a.ticket + 1, 1u);
  for (int it = 0, g = gwarp;; ++it) {
    if (it < static_rounds) {
      g = gwarp + it * gwarps;
    } else {
      g = n_static + __shfl_sync(~0u, g_next, 0);
      if (g >= ngroups) break;
      if (lane == 0) g_next = (int)atomicAdd(a.ticket + 1, 1u);
    }
    process_group(g);
  }

  // ---- CTA merge: the warps' sorted lists are merged in registers into
  // warp 0 (cta_merge_lists), which publishes the k best; warp 0 also folds
  // the warps' (max, sumexp).
  float* rec[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    // the workspace holds kHeadMaxCtas records per hidden state (a failed
    // check in a debug build writes record 0 instead)
    rec[m] = a.part + (VT_CHECKED(gridDim.x <= kHeadMaxCtas)
                           ? ((size_t)m * gridDim.x + blockIdx.x) * a.pstride
                           : 0);
    if (lane == 0) { w_mx[m][warp] = mx[m]; w_se[m][warp] = se[m]; }
  }
  int level = 0;
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    entry_key x = tk[m];
    int y = __float_as_int(ts[m]);
    cta_merge_lists<kGemvWarps, kSample>(x, y, msc.slots, level);
    if (warp == 0) {
      if (lane < k) {
        reinterpret_cast<entry_key*>(rec[m] + 4)[lane] = x;
        if (kSample) rec[m][4 + 2 * k + lane] = __int_as_float(y);
      }
      const float wmx = lane < kGemvWarps ? w_mx[m][lane] : -INFINITY;
      const float wse = lane < kGemvWarps ? w_se[m][lane] : 0.f;
      float M_b = wmx;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M_b = fmaxf(M_b, __shfl_xor_sync(~0u, M_b, o));
      float S_b = wse > 0.f ? wse * __expf(wmx - M_b) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) S_b += __shfl_xor_sync(~0u, S_b, o);
      if (lane == 0) { rec[m][0] = M_b; rec[m][1] = S_b; }
    }
  }

  // ---- last CTA merges every CTA's (max, sumexp, top-k).  The barrier
  // orders the CTA's partial writes before thread 0's gpu-scope release on
  // the ticket; the last arrival's acquire (and the barrier after it) makes
  // every CTA's partials visible to the whole merging CTA.
  __syncthreads();
  if (tid == 0) s_last = ticket_arrive(a.ticket) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  head_final_merge<kGemvThreads>(a, MR, gridDim.x, hs, msc, &merge_bar);
  if (tid == 0) {
    a.ticket[0] = 0u;
    a.ticket[1] = 0u;
  }
}

template <int MR, int CPL, int U, bool kSample>
vt_status launch_gemv(const HeadArgs& a, const DeviceInfo& di,
                      cudaStream_t s) {
  auto kern = head_gemv_kernel<MR, CPL, U, kSample>;
  const int64_t groups = (a.V_high + U - 1) / U;
  // One CTA per SM (the launch bound); no more CTAs than warps have rows,
  // and no more than the last CTA can stage records of.
  int64_t G = std::min<int64_t>((int64_t)di.num_sms,
                                (groups + kGemvWarps - 1) / kGemvWarps);
  G = std::min<int64_t>(G, kStageBytesMax / (a.pstride * (int64_t)sizeof(float)));
  G = std::max<int64_t>(1, std::min<int64_t>(G, kHeadMaxCtas));
  const int smem = (int)std::max<int64_t>((int64_t)MR * a.d * sizeof(float),
                                          G * a.pstride * (int64_t)sizeof(float));
  if (smem > di.max_smem_optin)
    return fail(VT_ERR_UNSUPPORTED, "head_gemv: M * d too large for smem");
  if (!allow_max_smem(kern, di)) return VT_ERR_CUDA;
  const cudaError_t e =
      launch_dependent(kern, dim3((unsigned)G), dim3(kGemvThreads), smem, s, a);
  if (e != cudaSuccess)
    return fail(VT_ERR_CUDA, std::string("head_gemv_kernel: ") + cudaGetErrorString(e));
  return launch_status("head_gemv_kernel");
}

// U rows per warp step: enough 16-byte loads in flight per lane (U * CPL up
// to 16) without the accumulators (U * MR) spilling.
template <int MR, int CPL>
vt_status launch_cpl(const HeadArgs& a, const DeviceInfo& di, cudaStream_t s) {
  constexpr int U0 = 16 / CPL < 8 / MR ? 16 / CPL : 8 / MR;
  constexpr int U = U0 < 1 ? 1 : U0;
  return a.opt.sample ? launch_gemv<MR, CPL, U, true>(a, di, s)
                      : launch_gemv<MR, CPL, U, false>(a, di, s);
}

template <int MR>
vt_status dispatch_cpl(const HeadArgs& a, const DeviceInfo& di,
                       cudaStream_t s) {
  const int nchunks = a.d / 8;
  if (nchunks <= 32) return launch_cpl<MR, 1>(a, di, s);
  if (nchunks <= 64) return launch_cpl<MR, 2>(a, di, s);
  if (nchunks <= 128) return launch_cpl<MR, 4>(a, di, s);
  // Wider rows stream as two rows of 8 chunks a lane per step (two half
  // rows in flight per warp), not one whole row of 16: measured 41.7 against
  // 49.0 us at d = 4096, V_high = 32768.
  return launch_cpl<MR, 8>(a, di, s);
}

}  // namespace

vt_status head_gemv(const HeadArgs& a, const DeviceInfo& di, cudaStream_t s) {
  switch (a.M) {
    case 1: return dispatch_cpl<1>(a, di, s);
    case 2: return dispatch_cpl<2>(a, di, s);
    case 3: return dispatch_cpl<3>(a, di, s);
    case 4: return dispatch_cpl<4>(a, di, s);
    default: return fail(VT_ERR_UNSUPPORTED, "head_gemv: M > 4");
  }
}

}  // namespace vt
