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
#include "vt_checks.cuh"
#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kCountThreads = 1024;
constexpr int kCountMaxCtas = 256;               // workspace is sized for this
constexpr int64_t kTokensPerCta = 1 << 17;       // below this, fewer CTAs
constexpr int kCountMaxIds = 208 * 1024;         // ids per pass (bytes of smem)

// Byte wraps (and the carries they push into the next byte of the word)
// are settled in 32-bit counters.  Wraps come from frequent ids, so a small
// shared-memory table (kCacheSlots direct-mapped slots, tagged with the id,
// claimed by compare-and-swap) holds those counters for the hot ids and is
// added to the global counts once at the end; an id whose slot is taken by
// another id goes to the global counts directly.  This keeps the hottest
// ids from receiving one global atomic per 256 hits from every CTA.
constexpr int kCacheSlots = 2048;
constexpr uint32_t kEmptyTag = 0xffffffffu;

struct WrapCache {
  uint32_t tag[kCacheSlots];
  uint32_t cnt[kCacheSlots];
};

__device__ __forceinline__ void cache_add(WrapCache& wc, uint32_t u,
                                          uint32_t delta, uint32_t* counts) {
  const uint32_t slot = u & (kCacheSlots - 1);
  uint32_t t = wc.tag[slot];
  if (t == kEmptyTag) {
    const uint32_t prev = atomicCAS(&wc.tag[slot], kEmptyTag, u);
    t = prev == kEmptyTag ? u : prev;
  }
  if (t == u) atomicAdd(&wc.cnt[slot], delta);
  else atomicAdd(&counts[u], delta);
}

// The hit that made byte b0 of shared word `word` wrap (old byte 0xff):
// +256 for that id; the carry added 1 to the next byte, so -1 for the next
// id, which may itself have wrapped (+256), and so on along the word.
__device__ __noinline__ void settle_wrap(uint32_t old, uint32_t word,
                                         uint32_t b0, uint32_t* counts,
                                         uint32_t Vr, WrapCache& wc) {
  const uint32_t base = word << 2;
  if (!VT_CHECKED(base + b0 < Vr)) return;
  cache_add(wc, base + b0, 256u, counts);
  for (uint32_t b = b0 + 1; b < 4; ++b) {
    if (base + b >= Vr) break;  // padding byte: never counted, never reported
    const uint32_t ob = (old >> (8 * b)) & 0xffu;
    if (ob == 0xffu) {
      cache_add(wc, base + b, 255u, counts);  // carry in (-1) and a wrap (+256)
    } else {
      cache_add(wc, base + b, 0xffffffffu, counts);  // carry in only: -1
      break;
    }
  }
}

// Pass kinds.  kPadded: one pass over every id with V % 4 == 0; an id
// outside 0..V-1 is clamped to V, byte 0 of a padding word after the
// histogram, so a token needs no validity test or select: the padding
// byte's hits (256 per wrap plus its final value) are the invalid tokens.
// kSingle: one pass over every id, V % 4 != 0.  kRange: one of several
// passes over id ranges (ids outside the range belong to other passes).
constexpr int kPadded = 0, kSingle = 1, kRange = 2;

// Sixteen tokens of one thread.  The sixteen shared-memory atomics issue
// back to back (their latencies overlap); a token's byte wrapped if its old
// value was 0xff, and the checks fold into one bit mask, so the rare wraps
// (once per 256 hits of an id) cost one branch per 16 tokens.  An id this
// pass does not count adds 0 (kSingle, kRange), which changes nothing.
template <int kMode>
__device__ __forceinline__ void count16(uint32_t* sm, const int4 (&v)[4],
                                        uint32_t lo, uint32_t Vr, uint32_t V,
                                        uint32_t* counts_pass,
                                        uint32_t& invalid, WrapCache& wc) {
  uint32_t t[16], olds[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    t[4 * q + 0] = (uint32_t)v[q].x;
    t[4 * q + 1] = (uint32_t)v[q].y;
    t[4 * q + 2] = (uint32_t)v[q].z;
    t[4 * q + 3] = (uint32_t)v[q].w;
  }
  uint32_t wraps = 0;  // bit j: token j's byte wrapped
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (kMode == kPadded) {
      const uint32_t u = min(t[j], Vr);
      const uint32_t sh = (u & 3u) << 3;
      olds[j] = atomicAdd(&sm[u >> 2], 1u << sh);
      if (((olds[j] >> sh) & 0xffu) == 0xffu) wraps |= 1u << j;
    } else {
      const uint32_t u = kMode == kSingle ? t[j] : t[j] - lo;
      const bool in = u < Vr;
      const uint32_t sh = (u & 3u) << 3;
      olds[j] = atomicAdd(&sm[in ? u >> 2 : 0u], in ? 1u << sh : 0u);
      if (in && ((olds[j] >> sh) & 0xffu) == 0xffu) wraps |= 1u << j;
      if (kMode == kSingle) invalid += in ? 0u : 1u;
      else if (lo == 0) invalid += t[j] >= V ? 1u : 0u;
    }
  }
  // A warp sees about two wraps per step of 512 tokens, so this loop runs
  // in most steps, but only over the wrapped tokens of each thread.
  while (wraps) {
    const int j = __ffs(wraps) - 1;
    wraps &= wraps - 1;
    uint32_t tj = 0, oj = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q)
      if (q == j) { tj = t[q]; oj = olds[q]; }
    const uint32_t u = kMode == kPadded ? min(tj, Vr)
                                        : (kMode == kSingle ? tj : tj - lo);
    if (kMode == kPadded && u == Vr) invalid += 256u;  // the padding byte
    else settle_wrap(oj, u >> 2, u & 3u, counts_pass, Vr, wc);
  }
}

// One token (loop tails).
__device__ __forceinline__ void count1(uint32_t* sm, uint32_t t, uint32_t lo,
                                       uint32_t Vr, uint32_t V,
                                       uint32_t* counts_pass,
                                       uint32_t& invalid, WrapCache& wc) {
  const uint32_t u = t - lo;
  if (u < Vr) {
    const uint32_t sh = (u << 3) & 24u;
    const uint32_t old = atomicAdd(&sm[u >> 2], 1u << sh);
    if (((old >> sh) & 0xffu) == 0xffu)
      settle_wrap(old, u >> 2, u & 3u, counts_pass, Vr, wc);
  } else if (lo == 0 && t >= V) {
    ++invalid;
  }
}

template <int kMode>
__global__ void __launch_bounds__(kCountThreads, 1)
    count_tokens_kernel(const int32_t* __restrict__ tokens, int64_t n,
                        uint32_t V, uint32_t lo, uint32_t Vr,
                        uint32_t* __restrict__ counts,
                        unsigned long long* __restrict__ n_invalid,
                        uint32_t* __restrict__ slabs, int words_padded) {
  extern __shared__ __align__(16) uint32_t sm[];
  __shared__ WrapCache wc;
  for (int i = threadIdx.x; i < words_padded; i += kCountThreads) sm[i] = 0;
  for (int i = threadIdx.x; i < kCacheSlots; i += kCountThreads) {
    wc.tag[i] = kEmptyTag;
    wc.cnt[i] = 0u;
  }
  __syncthreads();

  uint32_t* counts_pass = counts + lo;
  uint32_t invalid = 0;
  const int64_t n4 = n >> 2;
  const int4* t4 = reinterpret_cast<const int4*>(tokens);
  const int64_t stride = (int64_t)gridDim.x * kCountThreads;
  int64_t i = (int64_t)blockIdx.x * kCountThreads + threadIdx.x;
  // Steps of four int4 (16 tokens) per thread, two buffers in ping-pong:
  // the loads of the next step are in flight while this step counts.
  int4 a[4], b[4];
  auto load4 = [&](int4 (&dst)[4], int64_t at) {
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = ld_stream_i4(t4 + at + q * stride);
  };
  const int64_t step = 4 * stride;
  if (i + 3 * stride < n4) {
    load4(a, i);
    while (true) {
      const bool more_b = i + step + 3 * stride < n4;
      if (more_b) load4(b, i + step);
      count16<kMode>(sm, a, lo, Vr, V, counts_pass, invalid, wc);
      i += step;
      if (!more_b) break;
      const bool more_a = i + step + 3 * stride < n4;
      if (more_a) load4(a, i + step);
      count16<kMode>(sm, b, lo, Vr, V, counts_pass, invalid, wc);
      i += step;
      if (!more_a) break;
    }
  }
  for (; i < n4; i += stride) {
    const int4 x = ld_stream_i4(t4 + i);
    count1(sm, (uint32_t)x.x, lo, Vr, V, counts_pass, invalid, wc);
    count1(sm, (uint32_t)x.y, lo, Vr, V, counts_pass, invalid, wc);
    count1(sm, (uint32_t)x.z, lo, Vr, V, counts_pass, invalid, wc);
    count1(sm, (uint32_t)x.w, lo, Vr, V, counts_pass, invalid, wc);
  }
  if (blockIdx.x == 0 && threadIdx.x < (n & 3))
    count1(sm, (uint32_t)tokens[(n4 << 2) + threadIdx.x], lo, Vr, V,
           counts_pass, invalid, wc);
  __syncthreads();
  // kPadded: the padding byte's final value adds to the invalid tokens
  if (kMode == kPadded && threadIdx.x == 0) invalid += sm[Vr >> 2] & 0xffu;

  uint32_t* slab = slabs + (size_t)blockIdx.x * words_padded;
  if (VT_CHECKED(blockIdx.x < kCountMaxCtas))
    for (int w = threadIdx.x; w < words_padded; w += kCountThreads)
      slab[w] = sm[w];
  for (int i = threadIdx.x; i < kCacheSlots; i += kCountThreads)
    if (wc.tag[i] != kEmptyTag && wc.cnt[i] != 0u && VT_CHECKED(wc.tag[i] < Vr))
      atomicAdd(&counts_pass[wc.tag[i]], wc.cnt[i]);

  if (lo == 0 && n_invalid) {
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

// Histogram words of a pass over Vr ids: one byte per id plus (for a
// padded pass) the padding word at Vr / 4, rounded up to 16 bytes.
int words_for(uint32_t Vr) { return (int)((Vr / 4 + 1 + 3) & ~3u); }

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
  const int ids_per_pass = std::min<int>(
      kCountMaxIds, ((di.max_smem_optin - (int)sizeof(WrapCache)) / 16) * 16 - 16);
  if (!allow_max_smem(count_tokens_kernel<kPadded>, di) ||
      !allow_max_smem(count_tokens_kernel<kSingle>, di) ||
      !allow_max_smem(count_tokens_kernel<kRange>, di))
    return VT_ERR_CUDA;
  const int G = (int)std::max<int64_t>(
      1, std::min<int64_t>({(int64_t)di.num_sms, (int64_t)kCountMaxCtas,
                            (n + kTokensPerCta - 1) / kTokensPerCta}));
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* slabs = static_cast<uint32_t*>(ws);
  for (int64_t lo = 0; lo < V; lo += ids_per_pass) {
    const uint32_t Vr = (uint32_t)std::min<int64_t>(ids_per_pass, V - lo);
    const int words = words_for(Vr);
    const bool single = lo == 0 && Vr == (uint32_t)V;
    auto kern = !single ? count_tokens_kernel<kRange>
                : Vr % 4 == 0 ? count_tokens_kernel<kPadded>
                              : count_tokens_kernel<kSingle>;
    kern<<<G, kCountThreads, words * sizeof(uint32_t), s>>>(
        tokens, n, (uint32_t)V, (uint32_t)lo, Vr, counts,
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
