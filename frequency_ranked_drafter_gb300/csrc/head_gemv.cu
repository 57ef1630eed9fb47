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
// At M <= 4 hidden states the head is a GEMV bound by reading W_high once
// (V_high * d * 2 bytes).  One launch does everything:
//   * every warp of the grid streams whole rows of W_high with 16-byte
//     loads (up to 16 per lane in flight) and dots them with H, which each
//     CTA keeps in shared memory as fp32; rows are dealt round-robin over all
//     warps of the grid, so every SM streams the same number of bytes;
//   * each warp keeps, per hidden state, an online (max, sum of exp) and a
//     sorted top-k list held one entry per lane (insertion by ballot and a
//     one-lane shift), so no logit is ever written to memory;
//   * each CTA merges its warps' lists by rank counting in shared memory and
//     publishes (max, sumexp, top-k) to the workspace; the last CTA to finish
//     (atomic ticket, no waiting) merges all CTAs (head_final_merge),
//     rescales the sums, writes ids and probabilities and re-arms the ticket.
#include <float.h>

#include "head_common.cuh"

namespace vt {
namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;

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

template <int MR, int CPL, int U>
__global__ void __launch_bounds__(kGemvThreads, 2)
    head_gemv_kernel(HeadArgs a) {
  extern __shared__ __align__(16) float hs[];  // [MR][d] fp32 hidden states
  __shared__ float c_val[MR][kGemvWarps * kTopKMax];
  __shared__ int c_idx[MR][kGemvWarps * kTopKMax];
  __shared__ float w_mx[MR][kGemvWarps], w_se[MR][kGemvWarps];
  __shared__ MergeScratch msc;
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = a.d, k = a.k;

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

  float mx[MR], se[MR], tv[MR], thr[MR];
  int ti[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    mx[m] = -INFINITY; se[m] = 0.f; tv[m] = -INFINITY; thr[m] = -INFINITY;
    ti[m] = INT_MAX;
  }

  const int nchunks = d >> 3;
  const int nkb = (nchunks + 32 * CPL - 1) / (32 * CPL);
  const int gwarps = gridDim.x * kGemvWarps;
  const int gwarp = blockIdx.x * kGemvWarps + warp;
  const float4* h4 = reinterpret_cast<const float4*>(hs);
  const int ngroups = (a.V_high + U - 1) / U;

  auto process_group = [&](int g) {
    const int r0 = g * U;
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
        const float l = warp_sum(acc[u][m]);
        if (a.out_logits && lane == 0)
          a.out_logits[(int64_t)m * a.V_high + row] = l;
        if (l > mx[m]) {
          se[m] = se[m] * __expf(mx[m] - l) + 1.f;
          mx[m] = l;
        } else {
          se[m] += __expf(l - mx[m]);
        }
        // rows grow along a warp's walk, so an equal logit never displaces
        if (l > thr[m]) {
          const unsigned ahead = __ballot_sync(~0u, lane < k && tv[m] >= l);
          const int p = __popc(ahead);
          const float up_v = __shfl_up_sync(~0u, tv[m], 1);
          const int up_i = __shfl_up_sync(~0u, ti[m], 1);
          if (lane == p) { tv[m] = l; ti[m] = row; }
          else if (lane > p && lane < k) { tv[m] = up_v; ti[m] = up_i; }
          thr[m] = __shfl_sync(~0u, tv[m], k - 1);
        }
      }
    }
  };

  // Rows are dealt in groups of U.  Most groups go round-robin over all
  // warps of the grid; the last ~1/8 are handed out one at a time from a
  // global counter, so warps that stream faster take more and all warps
  // finish together.  A warp asks for its next dynamic group one group ahead.
  const int static_rounds = (ngroups / gwarps) * 7 / 8;
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

  // ---- CTA merge: rank counting over the warps' lists.
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    if (lane < k) {
      c_val[m][warp * k + lane] = tv[m];
      c_idx[m][warp * k + lane] = ti[m];
    }
    if (lane == 0) { w_mx[m][warp] = mx[m]; w_se[m][warp] = se[m]; }
  }
  __syncthreads();
  const int nc = kGemvWarps * k;
  float* part = a.part + (size_t)blockIdx.x * MR * a.pstride;
  for (int t = tid; t < MR * a.pstride; t += kGemvThreads) {
    // empty slots of the published list: (-inf, INT_MAX)
    const int o = t % a.pstride;
    if (o >= 2 && o < 2 + k) part[t] = -INFINITY;
    else if (o >= 2 + k && o < 2 + 2 * k) reinterpret_cast<int*>(part)[t] = INT_MAX;
  }
  __syncthreads();
  for (int t = tid; t < MR * nc; t += kGemvThreads) {
    const int m = t / nc, c = t % nc;
    const float v = c_val[m][c];
    const int i = c_idx[m][c];
    if (i == INT_MAX) continue;
    int rank = 0;
    for (int q = 0; q < nc; ++q) rank += key_beats(c_val[m][q], c_idx[m][q], v, i);
    if (rank < k) {
      part[m * a.pstride + 2 + rank] = v;
      reinterpret_cast<int*>(part)[m * a.pstride + 2 + k + rank] = i;
    }
  }
  if (tid < MR) {
    const int m = tid;
    float M_b = -INFINITY;
    for (int w = 0; w < kGemvWarps; ++w) M_b = fmaxf(M_b, w_mx[m][w]);
    float S_b = 0.f;
    for (int w = 0; w < kGemvWarps; ++w)
      if (w_se[m][w] > 0.f) S_b += w_se[m][w] * __expf(w_mx[m][w] - M_b);
    part[m * a.pstride + 0] = M_b;
    part[m * a.pstride + 1] = S_b;
  }

  // ---- last CTA merges every CTA's (max, sumexp, top-k).  The barrier
  // orders the CTA's partial writes before thread 0's gpu-scope release on
  // the ticket; the last arrival's acquire (and the barrier after it) makes
  // every CTA's partials visible to the whole merging CTA.
  __syncthreads();
  if (tid == 0) s_last = ticket_arrive(a.ticket) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  head_final_merge<kGemvThreads>(a, MR, gridDim.x, hs, msc);
  if (tid == 0) {
    a.ticket[0] = 0u;
    a.ticket[1] = 0u;
  }
}

template <int MR, int CPL, int U>
vt_status launch_gemv(const HeadArgs& a, const DeviceInfo& di,
                      cudaStream_t s) {
  auto kern = head_gemv_kernel<MR, CPL, U>;
  const int64_t groups = (a.V_high + U - 1) / U;
  // Two CTAs per SM (the launch bound); no more CTAs than warps have rows,
  // and no more than the last CTA can stage candidates of (G * k * 8 bytes).
  int64_t G = std::min<int64_t>((int64_t)di.num_sms * 2,
                                (groups + kGemvWarps - 1) / kGemvWarps);
  G = std::min<int64_t>(G, kStageBytesMax / (8 * a.k));
  G = std::max<int64_t>(1, std::min<int64_t>(G, kHeadMaxCtas));
  const int smem = (int)std::max<int64_t>((int64_t)MR * a.d * sizeof(float),
                                          G * a.k * 8);
  if (smem > di.max_smem_optin)
    return fail(VT_ERR_UNSUPPORTED, "head_gemv: M * d too large for smem");
  if (!allow_max_smem(kern, di)) return VT_ERR_CUDA;
  kern<<<(int)G, kGemvThreads, smem, s>>>(a);
  return launch_status("head_gemv_kernel");
}

// U rows per warp step: enough 16-byte loads in flight per lane (U * CPL up
// to 16) without the accumulators (U * MR) spilling.
template <int MR, int CPL>
vt_status launch_cpl(const HeadArgs& a, const DeviceInfo& di, cudaStream_t s) {
  constexpr int U0 = 16 / CPL < 8 / MR ? 16 / CPL : 8 / MR;
  constexpr int U = U0 < 1 ? 1 : U0;
  return launch_gemv<MR, CPL, U>(a, di, s);
}

template <int MR>
vt_status dispatch_cpl(const HeadArgs& a, const DeviceInfo& di,
                       cudaStream_t s) {
  const int nchunks = a.d / 8;
  if (nchunks <= 32) return launch_cpl<MR, 1>(a, di, s);
  if (nchunks <= 64) return launch_cpl<MR, 2>(a, di, s);
  if (nchunks <= 128) return launch_cpl<MR, 4>(a, di, s);
  if (nchunks <= 256) return launch_cpl<MR, 8>(a, di, s);
  return launch_cpl<MR, 16>(a, di, s);
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
