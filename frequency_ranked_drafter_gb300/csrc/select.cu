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
// (count desc, id asc) key without ever forming it.
//   * one kernel builds the digit histograms of all four passes at once
//     (a pass's totals do not depend on the order of the elements);
//   * one kernel per pass ("onesweep"): a CTA takes the next tile of 1024
//     elements, ranks them stably by digit in one round (warp match_any
//     plus a parallel prefix over the 32 warps), publishes its digit counts
//     and finds the counts of all earlier tiles by decoupled look-back
//     (each earlier tile publishes an aggregate first and an inclusive
//     prefix once it knows its own), then scatters.  Tiles are numbered in
//     the order their CTAs start, so a look-back only waits on tiles that
//     are already running; every wait is bounded and a wait that gives up
//     writes VT_ERR_TIMEOUT to the workspace error word;
//   * the last pass writes t2f, f2t and the two sums instead of a copy.
// About 1 MB of data at V = 128256: the cost is latency, not bandwidth.
#include "vt_checks.cuh"
#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kSelThreads = 1024;  // one element per thread per tile
constexpr int kSelTile = kSelThreads;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxV = 1 << 24;
constexpr int kHistThreads = 1024;
constexpr long long kLookbackBudget = 2000000000LL;  // about a second
constexpr int kLookback = 8;  // predecessor tiles read per look-back step
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagIncl = 2u << 30;
constexpr uint32_t kValMask = (1u << 30) - 1u;

__device__ __forceinline__ uint32_t digit_of(uint32_t key, int shift) {
  return 255u - ((key >> shift) & 255u);  // ascending digit = descending count
}

// A tile's status word carries its flag and its count in one 32-bit store,
// and nothing else is read on its strength, so relaxed gpu-scope accesses
// suffice (and let a window of look-back loads overlap).
__device__ __forceinline__ void st_status(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_status(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Digit histograms of the four passes: ghist[pass][digit] (zeroed by the
// caller).  Also zeroes the output sums, which the last pass accumulates.
__global__ void __launch_bounds__(kHistThreads)
    digits_hist_kernel(const uint32_t* __restrict__ counts, int V,
                       uint32_t* __restrict__ ghist,
                       unsigned long long* __restrict__ sums) {
  __shared__ uint32_t h[4 * 256];
  for (int i = threadIdx.x; i < 4 * 256; i += kHistThreads) h[i] = 0;
  __syncthreads();
  for (int e = blockIdx.x * kHistThreads + threadIdx.x; e < V;
       e += gridDim.x * kHistThreads) {
    const uint32_t c = counts[e];
#pragma unroll
    for (int p = 0; p < 4; ++p) atomicAdd(&h[p * 256 + digit_of(c, 8 * p)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 4 * 256; i += kHistThreads)
    if (h[i]) atomicAdd(&ghist[i], h[i]);
  if (blockIdx.x == 0 && threadIdx.x < 2) sums[threadIdx.x] = 0ull;
}

struct PassArgs {
  const uint32_t* keys_in;
  const int32_t* vals_in;  // null: the element index (first pass)
  uint32_t* keys_out;
  int32_t* vals_out;
  int V, shift;
  const uint32_t* ghist;  // this pass's 256 digit totals
  uint32_t* status;       // [tiles][256], zero before the pass
  uint32_t* tile_counter;
  unsigned* err;
  int final_pass, V_high;
  int32_t* t2f;
  int32_t* f2t;
  unsigned long long* sums;
};

__global__ void __launch_bounds__(kSelThreads, 1) onesweep_kernel(PassArgs a) {
  __shared__ uint32_t s_tile;
  __shared__ uint32_t dstart[256];  // first output slot of each digit
  __shared__ uint32_t tcnt[256];    // this tile's digit counts
  __shared__ uint32_t base[256];    // output slot of this tile's first element per digit
  __shared__ uint32_t wcnt[kSelWarps][256];
  __shared__ unsigned long long red[2][kSelWarps];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;

  if (t == 0) s_tile = atomicAdd(a.tile_counter, 1u);
  for (int i = t; i < kSelWarps * 256; i += kSelThreads) (&wcnt[0][0])[i] = 0u;
  __syncthreads();
  const uint32_t tile = s_tile;
  const int e = (int)tile * kSelTile + t;
  const bool valid = e < a.V;
  const uint32_t key = valid ? a.keys_in[e] : 0u;
  const int32_t val = valid ? (a.vals_in ? a.vals_in[e] : e) : 0;
  const uint32_t dig = valid ? digit_of(key, a.shift) : 256u;
  const unsigned peers = __match_any_sync(~0u, dig);
  const uint32_t rk = __popc(peers & lt_mask);
  if (valid && rk == 0) wcnt[warp][dig] = __popc(peers);
  __syncthreads();
  {  // per digit, an exclusive prefix over the 32 warps and the tile total:
     // thread t handles digit t/4 and warps 8*(t%4) .. 8*(t%4)+7
    const uint32_t d = t >> 2, part = t & 3;
    uint32_t c[8], run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) { c[j] = wcnt[8 * part + j][d]; run += c[j]; }
    uint32_t inc = run;
    const uint32_t y1 = __shfl_up_sync(~0u, inc, 1);
    if (part >= 1) inc += y1;
    const uint32_t y2 = __shfl_up_sync(~0u, inc, 2);
    if (part >= 2) inc += y2;
    uint32_t ex = inc - run;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      wcnt[8 * part + j][d] = ex;
      ex += c[j];
    }
    if (part == 3) tcnt[d] = inc;
  }
  __syncthreads();

  if (t < 256) {  // decoupled look-back, one digit per thread
    const uint32_t d = t, mine = tcnt[d];
    uint32_t* st = a.status + (size_t)tile * 256;
    uint32_t excl = 0;
    if (tile == 0) {
      st_status(&st[d], kFlagIncl | mine);
    } else {
      st_status(&st[d], kFlagAgg | mine);
      // walk back over earlier tiles, kLookback at a time: the loads of a
      // window are issued together, then read nearest first
      int j = (int)tile - 1;
      long long t0 = 0;
      bool waited = false, done = false;
      while (!done && j >= 0) {
        uint32_t w[kLookback];
#pragma unroll
        for (int q = 0; q < kLookback; ++q)
          w[q] = j - q >= 0 ? ld_status(&a.status[(size_t)(j - q) * 256 + d]) : kFlagIncl;
        int q = 0;
        for (; q < kLookback && j - q >= 0; ++q) {
          const uint32_t flag = w[q] & ~kValMask;
          if (flag == 0u) break;  // not published yet: reload from here
          excl += w[q] & kValMask;
          if (flag == kFlagIncl) { done = true; break; }
        }
        if (done) break;
        if (q < kLookback && j - q >= 0) {  // stopped on an unpublished tile
          if (!waited) { t0 = clock64(); waited = true; }
          if (clock64() - t0 > kLookbackBudget) {
            atomicExch(a.err, (unsigned)VT_ERR_TIMEOUT);
            break;
          }
        }
        j -= q;
      }
      st_status(&st[d], kFlagIncl | (excl + mine));
    }
    base[d] = excl;
  } else if (t < 288) {  // meanwhile: exclusive scan of the digit totals
    const int l = t - 256;
    uint32_t v[8], run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) { v[j] = a.ghist[8 * l + j]; run += v[j]; }
    uint32_t inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(~0u, inc, o);
      if (l >= o) inc += y;
    }
    uint32_t ex = inc - run;
#pragma unroll
    for (int j = 0; j < 8; ++j) { dstart[8 * l + j] = ex; ex += v[j]; }
  }
  __syncthreads();

  unsigned long long kept = 0, total = 0;
  if (valid) {
    const uint32_t pos = dstart[dig] + base[dig] + wcnt[warp][dig] + rk;
    if (a.final_pass) {
      if ((int)pos < a.V_high) {
        if (VT_CHECKED(val >= 0 && val < a.V)) {
          a.t2f[pos] = val;
          a.f2t[val] = (int32_t)pos;
        }
        kept = key;
      } else if (VT_CHECKED(val >= 0 && val < a.V)) {
        a.f2t[val] = -1;
      }
      total = key;
    } else if (VT_CHECKED(pos < (uint32_t)a.V)) {
      a.keys_out[pos] = key;
      a.vals_out[pos] = val;
    }
  }
  if (a.final_pass) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kept += __shfl_xor_sync(~0u, kept, o);
      total += __shfl_xor_sync(~0u, total, o);
    }
    if (lane == 0) { red[0][warp] = kept; red[1][warp] = total; }
    __syncthreads();
    if (t == 0) {
      unsigned long long x = 0, y = 0;
      for (int w = 0; w < kSelWarps; ++w) { x += red[0][w]; y += red[1][w]; }
      atomicAdd(&a.sums[0], x);
      atomicAdd(&a.sums[1], y);
    }
  }
}

// Workspace: a zero-initialised block (a 256-byte header whose 32-bit word
// at byte 128 is the error word, as in the head's workspace; digit
// histograms; per-pass tile status; tile counters) that one memset clears
// at the start of every call, then the keys/values ping-pong.
struct SelectLayout {
  size_t zero_begin, err, ghist, status, counters, zero_end, keys_a, vals_a,
      keys_b, vals_b, total;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

SelectLayout select_layout(int V) {
  const size_t T = (size_t)(V + kSelTile - 1) / kSelTile;
  SelectLayout L;
  size_t o = 0;
  L.zero_begin = o;
  L.err = o + 128; o += 256;
  L.ghist = o;    o += round256(4 * 256 * 4);
  L.status = o;   o += round256(4 * T * 256 * 4);
  L.counters = o; o += 256;
  L.zero_end = o;
  L.keys_a = o; o += round256((size_t)V * 4);
  L.vals_a = o; o += round256((size_t)V * 4);
  L.keys_b = o; o += round256((size_t)V * 4);
  L.vals_b = o; o += round256((size_t)V * 4);
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
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  char* base = static_cast<char*>(ws);
  uint32_t* keys[2] = {reinterpret_cast<uint32_t*>(base + L.keys_a),
                       reinterpret_cast<uint32_t*>(base + L.keys_b)};
  int32_t* vals[2] = {reinterpret_cast<int32_t*>(base + L.vals_a),
                      reinterpret_cast<int32_t*>(base + L.vals_b)};
  uint32_t* ghist = reinterpret_cast<uint32_t*>(base + L.ghist);
  uint32_t* status = reinterpret_cast<uint32_t*>(base + L.status);
  uint32_t* counters = reinterpret_cast<uint32_t*>(base + L.counters);
  auto* s64 = reinterpret_cast<unsigned long long*>(sums);
  const int T = (V + kSelTile - 1) / kSelTile;
  cudaStream_t s = (cudaStream_t)stream;

  if (cudaMemsetAsync(base + L.zero_begin, 0, L.zero_end - L.zero_begin, s) !=
      cudaSuccess)
    return launch_status("cudaMemsetAsync(select workspace)");
  // few CTAs with many elements each: fewer global atomics on the bins
  const int hb = std::max(1, std::min((V + 4 * kHistThreads - 1) / (4 * kHistThreads), 32));
  digits_hist_kernel<<<hb, kHistThreads, 0, s>>>(counts, V, ghist, s64);
  vt_status st = launch_status("digits_hist_kernel");
  if (st != VT_OK) return st;

  const uint32_t* kin = counts;
  const int32_t* vin = nullptr;  // pass 0: values are the ids themselves
  for (int pass = 0; pass < 4; ++pass) {
    PassArgs a;
    a.keys_in = kin;
    a.vals_in = vin;
    a.keys_out = pass < 3 ? keys[pass & 1] : nullptr;
    a.vals_out = pass < 3 ? vals[pass & 1] : nullptr;
    a.V = V;
    a.shift = 8 * pass;
    a.ghist = ghist + 256 * pass;
    a.status = status + (size_t)pass * T * 256;
    a.tile_counter = counters + pass;
    a.err = reinterpret_cast<unsigned*>(base + L.err);
    a.final_pass = pass == 3;
    a.V_high = V_high;
    a.t2f = t2f;
    a.f2t = f2t;
    a.sums = s64;
    onesweep_kernel<<<T, kSelThreads, 0, s>>>(a);
    st = launch_status("onesweep_kernel");
    if (st != VT_OK) return st;
    kin = a.keys_out;
    vin = a.vals_out;
  }
  return VT_OK;
}
