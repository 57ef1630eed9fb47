// vt_count_tokens — token-frequency histogram over a token stream.
//
// "VocabTrim: Memory-Efficient Vocabulary Pruning for Speculative Decoding",
// Implementation Step 1 (count every id into a dict) and "FR-Spec: ...
// Frequency-Ranked Speculative Sampling", Method > Key design (token
// frequencies over a 1B-token corpus subset).
//
// Design (one pass over HBM, 4 bytes per token):
//   * Each CTA keeps a private histogram of the whole id range in shared
//     memory with ONE BYTE per id (128256 ids -> 125 KB), four ids per
//     32-bit word.  A hit on id u adds 1 << 8*(u & 3) to word u >> 2 with a
//     shared-memory atomic.
//   * A byte wraps every 256 hits.  The atomic returns the old word, so the
//     thread that made a byte wrap knows it (its old byte was 0xFF) and
//     settles the wrap exactly in the global counts: +256 for the wrapped id,
//     and, because the wrap carried +1 into the next byte of the word,
//     -1 for the next id (+256 more if that byte wrapped as well, and so on).
//     With X wraps of a byte, C carries into it and final byte B, the id's
//     count is 256*X - C + B, which is exactly its number of hits.
//   * At the end each CTA writes its bytes to a per-CTA slab of the
//     workspace; a second kernel adds the slabs (four bytes at a time, in
//     16-bit SIMD lanes) into the uint32 counts.
//   * Vocabularies larger than the shared-memory byte budget are counted in
//     several passes over id ranges (the stream is re-read per pass).
#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kCountThreads = 1024;
constexpr int kCountMaxCtas = 256;               // workspace is sized for this
constexpr int64_t kTokensPerCta = 1 << 17;       // below this, fewer CTAs
constexpr int kCountMaxIds = 224 * 1024;         // ids per pass (bytes of smem)

__device__ __noinline__ void settle_wrap(uint32_t old, uint32_t word,
                                         uint32_t b0, uint32_t* counts,
                                         uint32_t Vr) {
  const uint32_t base = word << 2;
  atomicAdd(&counts[base + b0], 256u);  // byte b0 wrapped once
  for (uint32_t b = b0 + 1; b < 4; ++b) {
    if (base + b >= Vr) break;  // padding byte: never counted, never reported
    const uint32_t ob = (old >> (8 * b)) & 0xffu;
    if (ob == 0xffu) {
      atomicAdd(&counts[base + b], 255u);  // carry in (-1) and a wrap (+256)
    } else {
      atomicAdd(&counts[base + b], 0xffffffffu);  // carry in only: -1
      break;
    }
  }
}

// Counts one token whose word / shift are known; returns the old word.
__device__ __forceinline__ uint32_t smem_hit(uint32_t* sm, uint32_t u) {
  return atomicAdd(&sm[u >> 2], 1u << ((u & 3u) << 3));
}

// Eight tokens: all shared-memory atomics are issued back to back, and the
// (rare) byte wraps are settled afterwards, so the atomics' latencies
// overlap instead of each one gating a branch.
__device__ __forceinline__ void count8(uint32_t* sm, const int32_t (&t)[8],
                                       uint32_t lo, uint32_t Vr, uint32_t V,
                                       bool ci, uint32_t* counts_pass,
                                       uint32_t& invalid) {
  uint32_t old[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t u = static_cast<uint32_t>(t[j]) - lo;
    old[j] = 0;
    if (u < Vr) old[j] = smem_hit(sm, u);
    else if (ci && static_cast<uint32_t>(t[j]) >= V) ++invalid;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t u = static_cast<uint32_t>(t[j]) - lo;
    if (u < Vr && ((old[j] >> ((u & 3u) << 3)) & 0xffu) == 0xffu)
      settle_wrap(old[j], u >> 2, u & 3u, counts_pass, Vr);
  }
}

__device__ __forceinline__ void count1(uint32_t* sm, int32_t t, uint32_t lo,
                                       uint32_t Vr, uint32_t V, bool ci,
                                       uint32_t* counts_pass,
                                       uint32_t& invalid) {
  const uint32_t u = static_cast<uint32_t>(t) - lo;
  if (u < Vr) {
    const uint32_t old = smem_hit(sm, u);
    if (((old >> ((u & 3u) << 3)) & 0xffu) == 0xffu)
      settle_wrap(old, u >> 2, u & 3u, counts_pass, Vr);
  } else if (ci && static_cast<uint32_t>(t) >= V) {
    ++invalid;
  }
}

__global__ void __launch_bounds__(kCountThreads, 1)
    count_tokens_kernel(const int32_t* __restrict__ tokens, int64_t n,
                        uint32_t V, uint32_t lo, uint32_t Vr,
                        int count_invalid, uint32_t* __restrict__ counts,
                        unsigned long long* __restrict__ n_invalid,
                        uint32_t* __restrict__ slabs, int words_padded) {
  extern __shared__ __align__(16) uint32_t sm[];
  for (int i = threadIdx.x; i < words_padded; i += kCountThreads) sm[i] = 0;
  __syncthreads();

  uint32_t* counts_pass = counts + lo;
  uint32_t invalid = 0;
  const bool ci = count_invalid != 0;
  const int64_t n4 = n >> 2;
  const int4* t4 = reinterpret_cast<const int4*>(tokens);
  const int64_t stride = (int64_t)gridDim.x * kCountThreads;
  int64_t i = (int64_t)blockIdx.x * kCountThreads + threadIdx.x;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    const int4 a = ld_stream_i4(t4 + i);
    const int4 b = ld_stream_i4(t4 + i + stride);
    const int4 c = ld_stream_i4(t4 + i + 2 * stride);
    const int4 d = ld_stream_i4(t4 + i + 3 * stride);
    const int32_t x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    count8(sm, x, lo, Vr, V, ci, counts_pass, invalid);
    const int32_t y[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
    count8(sm, y, lo, Vr, V, ci, counts_pass, invalid);
  }
  for (; i < n4; i += stride) {
    const int4 a = ld_stream_i4(t4 + i);
    count1(sm, a.x, lo, Vr, V, ci, counts_pass, invalid);
    count1(sm, a.y, lo, Vr, V, ci, counts_pass, invalid);
    count1(sm, a.z, lo, Vr, V, ci, counts_pass, invalid);
    count1(sm, a.w, lo, Vr, V, ci, counts_pass, invalid);
  }
  if (blockIdx.x == 0 && threadIdx.x < (n & 3))
    count1(sm, tokens[(n4 << 2) + threadIdx.x], lo, Vr, V, ci, counts_pass,
           invalid);
  __syncthreads();

  uint32_t* slab = slabs + (size_t)blockIdx.x * words_padded;
  for (int w = threadIdx.x; w < words_padded; w += kCountThreads)
    slab[w] = sm[w];

  if (ci && n_invalid) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) invalid += __shfl_xor_sync(~0u, invalid, o);
    if ((threadIdx.x & 31) == 0 && invalid)
      atomicAdd(n_invalid, (unsigned long long)invalid);
  }
}

// counts[lo + 4w + b] += sum over CTAs of byte b of slab word w.  A CTA
// handles 32 words; its 8 warps each sum one eighth of the slabs with all
// loads of a thread issued together, and the eight partial sums are added
// in shared memory.  Bytes are summed in two registers of 16-bit lanes
// (at most 256 * 255 < 2^16).
constexpr int kReduceGroups = 8;
__global__ void __launch_bounds__(256)
    count_reduce_kernel(const uint32_t* __restrict__ slabs, int G,
                        int words_padded, uint32_t Vr,
                        uint32_t* __restrict__ counts_pass) {
  __shared__ uint32_t part[kReduceGroups][32][2];
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const uint32_t w = blockIdx.x * 32 + lane;
  const uint32_t nwords = (Vr + 3) / 4;
  uint32_t even = 0, odd = 0;  // bytes 0,2 and 1,3 of every slab word
  if (w < nwords) {
    constexpr int kPer = kCountMaxCtas / kReduceGroups;  // 32 slabs max
    uint32_t x[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = grp + j * kReduceGroups;
      x[j] = b < G ? __ldcg(slabs + (size_t)b * words_padded + w) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      even += x[j] & 0x00ff00ffu;
      odd += (x[j] >> 8) & 0x00ff00ffu;
    }
  }
  part[grp][lane][0] = even;
  part[grp][lane][1] = odd;
  __syncthreads();
  if (grp == 0 && w < nwords) {
    for (int g = 1; g < kReduceGroups; ++g) {
      even += part[g][lane][0];
      odd += part[g][lane][1];
    }
    const uint32_t s4[4] = {even & 0xffffu, odd & 0xffffu, even >> 16,
                            odd >> 16};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (4 * w + j < Vr) counts_pass[4 * w + j] += s4[j];
  }
}

int words_for(uint32_t Vr) { return (int)(((Vr + 3) / 4 + 3) & ~3u); }

}  // namespace
}  // namespace vt

extern "C" size_t vt_count_tokens_workspace_size(int32_t V) {
  if (V <= 0) return 0;
  const uint32_t Vr = (uint32_t)std::min<int64_t>(V, vt::kCountMaxIds);
  return (size_t)vt::kCountMaxCtas * vt::words_for(Vr) * sizeof(uint32_t);
}

extern "C" vt_status vt_count_tokens(const int32_t* tokens, int64_t n,
                                     int32_t V, uint32_t* counts,
                                     uint64_t* n_invalid, void* ws,
                                     size_t ws_bytes, void* stream) {
  using namespace vt;
  if (n < 0 || n >= (int64_t(1) << 40))
    return fail(VT_ERR_INVALID_ARG, "vt_count_tokens: need 0 <= n < 2^40");
  if (V <= 0 || V > (1 << 30))
    return fail(VT_ERR_INVALID_ARG, "vt_count_tokens: need 1 <= V <= 2^30");
  if (!counts || (n > 0 && !tokens))
    return fail(VT_ERR_INVALID_ARG, "vt_count_tokens: null pointer");
  if (tokens && !aligned(tokens, 16))
    return fail(VT_ERR_INVALID_ARG, "vt_count_tokens: tokens not 16B aligned");
  if (!ws || !aligned(ws, 256) || ws_bytes < vt_count_tokens_workspace_size(V))
    return fail(VT_ERR_WORKSPACE,
                "vt_count_tokens: workspace missing, misaligned or too small");
  if (n == 0) return VT_OK;
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  const int ids_per_pass =
      std::min<int>(kCountMaxIds, (di.max_smem_optin / 16) * 16);
  if (!allow_max_smem(count_tokens_kernel, di)) return VT_ERR_CUDA;
  const int G = (int)std::max<int64_t>(
      1, std::min<int64_t>({(int64_t)di.num_sms, (int64_t)kCountMaxCtas,
                            (n + kTokensPerCta - 1) / kTokensPerCta}));
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* slabs = static_cast<uint32_t*>(ws);
  for (int64_t lo = 0; lo < V; lo += ids_per_pass) {
    const uint32_t Vr = (uint32_t)std::min<int64_t>(ids_per_pass, V - lo);
    const int words = words_for(Vr);
    count_tokens_kernel<<<G, kCountThreads, words * sizeof(uint32_t), s>>>(
        tokens, n, (uint32_t)V, (uint32_t)lo, Vr, lo == 0, counts,
        reinterpret_cast<unsigned long long*>(n_invalid), slabs, words);
    vt_status st = launch_status("count_tokens_kernel");
    if (st != VT_OK) return st;
    const int rb = (int)(((Vr + 3) / 4 + 31) / 32);
    count_reduce_kernel<<<rb, 256, 0, s>>>(slabs, G, words, Vr, counts + lo);
    st = launch_status("count_reduce_kernel");
    if (st != VT_OK) return st;
  }
  return VT_OK;
}
