// vt_select_vocab — top-V_high selection by frequency and the two maps.
//
// "VocabTrim: Memory-Efficient Vocabulary Pruning for Speculative Decoding",
// Implementation Step 2: order ids by count (descending), keep the first
// target_vocab_size; an id's trimmed index is its rank in that order
// (full_to_trimmed / trimmed_to_full); coverage = selected / total count.
// Tie rule: lower id first, which makes the order a total order.
//
// Design: a stable least-significant-digit radix sort of the ids by count,
// descending, over four 8-bit digits.  The ids enter in ascending order and
// every pass is stable, so equal counts stay in ascending id order — the
// (count desc, id asc) key without ever forming it.  Each pass is two
// launches over tiles of 4096 elements: per-tile digit histograms, then a
// stable scatter (each CTA derives its own output offsets from all tiles'
// histograms).  The last scatter writes t2f, f2t and the two sums instead of
// another key/value copy.  The data is ~1 MB at V = 128256, so the cost is
// launch latency, not bandwidth.
#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelRounds = 16;
constexpr int kSelTile = kSelThreads * kSelRounds;  // 4096 elements
constexpr int kSelMaxV = 1 << 24;

__device__ __forceinline__ uint32_t digit_of(uint32_t key, int shift) {
  return 255u - ((key >> shift) & 255u);  // ascending digit = descending count
}

__global__ void __launch_bounds__(kSelThreads)
    radix_hist_kernel(const uint32_t* __restrict__ keys, int V, int shift,
                      uint32_t* __restrict__ tile_hist, int T,
                      unsigned long long* __restrict__ sums_to_zero) {
  __shared__ uint32_t h[256];
  h[threadIdx.x] = 0;
  __syncthreads();
  uint32_t key[kSelRounds];
#pragma unroll
  for (int r = 0; r < kSelRounds; ++r) {  // all loads first, then counting
    const int e = blockIdx.x * kSelTile + r * kSelThreads + threadIdx.x;
    key[r] = e < V ? keys[e] : 0u;
  }
#pragma unroll
  for (int r = 0; r < kSelRounds; ++r) {
    const int e = blockIdx.x * kSelTile + r * kSelThreads + threadIdx.x;
    if (e < V) atomicAdd(&h[digit_of(key[r], shift)], 1u);
  }
  __syncthreads();
  tile_hist[threadIdx.x * T + blockIdx.x] = h[threadIdx.x];
  if (sums_to_zero && blockIdx.x == 0 && threadIdx.x < 2)
    sums_to_zero[threadIdx.x] = 0ull;
}

// Block-wide exclusive scan of one value per thread (256 threads).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v,
                                                         uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(~0u, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  uint32_t before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  return before + inc - v;
}

template <bool kFinal>
__global__ void __launch_bounds__(kSelThreads)
    radix_scatter_kernel(const uint32_t* __restrict__ keys_in,
                         const int32_t* __restrict__ vals_in,  // null: e
                         int V, int shift,
                         const uint32_t* __restrict__ tile_hist, int T,
                         uint32_t* __restrict__ keys_out,
                         int32_t* __restrict__ vals_out, int V_high,
                         int32_t* __restrict__ t2f, int32_t* __restrict__ f2t,
                         unsigned long long* __restrict__ sums) {
  constexpr int kWarps = kSelThreads / 32;
  __shared__ uint32_t offs[256];
  __shared__ uint32_t wcnt[kWarps][257];  // column 256: out-of-range slots
  __shared__ uint32_t warp_tot[kWarps];
  __shared__ unsigned long long red[2][kWarps];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;

  // The tile's keys and values, loaded up front (round-major order).
  uint32_t keyr[kSelRounds];
  int32_t valr[kSelRounds];
#pragma unroll
  for (int r = 0; r < kSelRounds; ++r) {
    const int e = blockIdx.x * kSelTile + r * kSelThreads + t;
    keyr[r] = e < V ? keys_in[e] : 0u;
    valr[r] = e < V ? (vals_in ? vals_in[e] : e) : 0;
  }
  {  // output offset of digit t for this tile
    uint32_t total = 0, before = 0;
    for (int j0 = 0; j0 < T; j0 += 8) {
      uint32_t c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        c[j] = j0 + j < T ? tile_hist[t * T + j0 + j] : 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        total += c[j];
        if (j0 + j < (int)blockIdx.x) before += c[j];
      }
    }
    offs[t] = block_exclusive_scan(total, warp_tot) + before;
  }
  for (int w = 0; w < kWarps; ++w) wcnt[w][t] = 0;
  if (t < kWarps) wcnt[t][256] = 0;
  __syncthreads();

  unsigned long long kept = 0, total = 0;
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < kSelRounds; ++r) {
    const int e = blockIdx.x * kSelTile + r * kSelThreads + t;
    const bool valid = e < V;
    const uint32_t key = keyr[r];
    const int32_t val = valr[r];
    const uint32_t dig = valid ? digit_of(key, shift) : 256u;
    const unsigned peers = __match_any_sync(~0u, dig);
    const uint32_t rank = __popc(peers & lt_mask);
    if (rank == 0) wcnt[warp][dig] = __popc(peers);
    __syncthreads();
    if (valid) {
      uint32_t pos = offs[dig] + rank;
      for (int w = 0; w < warp; ++w) pos += wcnt[w][dig];
      if (kFinal) {
        if ((int)pos < V_high) {
          t2f[pos] = val;
          f2t[val] = (int32_t)pos;
          kept += key;
        } else {
          f2t[val] = -1;
        }
        total += key;
      } else {
        keys_out[pos] = key;
        vals_out[pos] = val;
      }
    }
    __syncthreads();
    uint32_t add = 0;
    for (int w = 0; w < kWarps; ++w) {
      add += wcnt[w][t];
      wcnt[w][t] = 0;
    }
    offs[t] += add;
    if (t < kWarps) wcnt[t][256] = 0;
    __syncthreads();
  }

  if (kFinal) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kept += __shfl_xor_sync(~0u, kept, o);
      total += __shfl_xor_sync(~0u, total, o);
    }
    if (lane == 0) {
      red[0][warp] = kept;
      red[1][warp] = total;
    }
    __syncthreads();
    if (t == 0) {
      unsigned long long a = 0, b = 0;
      for (int w = 0; w < kWarps; ++w) {
        a += red[0][w];
        b += red[1][w];
      }
      atomicAdd(&sums[0], a);
      atomicAdd(&sums[1], b);
    }
  }
}

struct SelectLayout {
  size_t keys_a, vals_a, keys_b, vals_b, hist, total;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

SelectLayout select_layout(int V) {
  const size_t T = (size_t)(V + kSelTile - 1) / kSelTile;
  SelectLayout L;
  size_t o = 0;
  L.keys_a = o; o += round256((size_t)V * 4);
  L.vals_a = o; o += round256((size_t)V * 4);
  L.keys_b = o; o += round256((size_t)V * 4);
  L.vals_b = o; o += round256((size_t)V * 4);
  L.hist = o;   o += round256(256 * T * 4);
  L.total = o;
  return L;
}

}  // namespace
}  // namespace vt

extern "C" size_t vt_select_vocab_workspace_size(int32_t V) {
  if (V <= 0) return 0;
  return vt::select_layout(V).total;
}

extern "C" vt_status vt_select_vocab(const uint32_t* counts, int32_t V,
                                     int32_t V_high, int32_t* t2f,
                                     int32_t* f2t, uint64_t* sums, void* ws,
                                     size_t ws_bytes, void* stream) {
  using namespace vt;
  if (!counts || !t2f || !f2t || !sums)
    return fail(VT_ERR_INVALID_ARG, "vt_select_vocab: null pointer");
  if (V <= 0 || V_high <= 0 || V_high > V)
    return fail(VT_ERR_INVALID_ARG,
                "vt_select_vocab: need 1 <= V_high <= V");
  if (V > kSelMaxV)
    return fail(VT_ERR_UNSUPPORTED, "vt_select_vocab: V > 2^24");
  if (!aligned(sums, 8))
    return fail(VT_ERR_INVALID_ARG, "vt_select_vocab: sums not 8B aligned");
  const SelectLayout L = select_layout(V);
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total)
    return fail(VT_ERR_WORKSPACE,
                "vt_select_vocab: workspace missing, misaligned or too small");
  char* base = static_cast<char*>(ws);
  uint32_t* keys[2] = {reinterpret_cast<uint32_t*>(base + L.keys_a),
                       reinterpret_cast<uint32_t*>(base + L.keys_b)};
  int32_t* vals[2] = {reinterpret_cast<int32_t*>(base + L.vals_a),
                      reinterpret_cast<int32_t*>(base + L.vals_b)};
  uint32_t* hist = reinterpret_cast<uint32_t*>(base + L.hist);
  auto* s64 = reinterpret_cast<unsigned long long*>(sums);
  const int T = (V + kSelTile - 1) / kSelTile;
  cudaStream_t s = (cudaStream_t)stream;

  const uint32_t* kin = counts;
  const int32_t* vin = nullptr;  // pass 0: values are the ids themselves
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    radix_hist_kernel<<<T, kSelThreads, 0, s>>>(kin, V, shift, hist, T,
                                                pass == 0 ? s64 : nullptr);
    vt_status st = launch_status("radix_hist_kernel");
    if (st != VT_OK) return st;
    if (pass < 3) {
      uint32_t* kout = keys[pass & 1];
      int32_t* vout = vals[pass & 1];
      radix_scatter_kernel<false><<<T, kSelThreads, 0, s>>>(
          kin, vin, V, shift, hist, T, kout, vout, V_high, nullptr, nullptr,
          nullptr);
      kin = kout;
      vin = vout;
    } else {
      radix_scatter_kernel<true><<<T, kSelThreads, 0, s>>>(
          kin, vin, V, shift, hist, T, nullptr, nullptr, V_high, t2f, f2t,
          s64);
    }
    st = launch_status("radix_scatter_kernel");
    if (st != VT_OK) return st;
  }
  return VT_OK;
}
