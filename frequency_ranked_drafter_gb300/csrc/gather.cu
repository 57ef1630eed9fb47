// vt_gather_rows / vt_gather_bias — reconstruction of the trimmed lm_head.
//
// "VocabTrim: Memory-Efficient Vocabulary Pruning for Speculative Decoding",
// Implementation Step 3: the trimmed weight is the original [vocab, hidden]
// weight indexed by trimmed_to_full along its rows, and an existing bias is
// indexed the same way.
//
// HBM-bound copy: every kept row (d bf16 = 2d bytes) is read once and written
// once.  One warp moves one row at a time with 16-byte loads; each lane keeps
// 8 loads in flight before its stores (4 KB per warp), with 32 warps resident
// per SM.  The grid is a whole number of waves over the SMs.
#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherChunks = 8;  // 16-byte chunks per lane per step

__global__ void __launch_bounds__(kGatherThreads, 4)
    gather_rows_kernel(const uint16_t* __restrict__ W, int64_t V, int d,
                       const int32_t* __restrict__ t2f, int V_high,
                       uint16_t* __restrict__ W_high,
                       unsigned long long* __restrict__ n_invalid) {
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (kGatherThreads / 32);
  const int warp = blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5);
  const int nchunks = d >> 3;  // 16-byte chunks per row
  for (int row = warp; row < V_high; row += warps_total) {
    const int64_t src = t2f[row];
    uint4* dst = reinterpret_cast<uint4*>(W_high + (int64_t)row * d);
    if (src < 0 || src >= V) {
      for (int c = lane; c < nchunks; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
      if (lane == 0 && n_invalid) atomicAdd(n_invalid, 1ull);
      continue;
    }
    const uint4* s = reinterpret_cast<const uint4*>(W + src * d);
    for (int base = 0; base < nchunks; base += 32 * kGatherChunks) {
      uint4 v[kGatherChunks];
#pragma unroll
      for (int j = 0; j < kGatherChunks; ++j) {
        const int c = base + lane + 32 * j;
        if (c < nchunks) v[j] = ld_stream_u4(s + c);
      }
#pragma unroll
      for (int j = 0; j < kGatherChunks; ++j) {
        const int c = base + lane + 32 * j;
        if (c < nchunks) st_stream_u4(dst + c, v[j]);
      }
    }
  }
}

// b_high[i] = b[t2f[i]]: one thread per kept id (a 1-D gather of 4-byte
// values, V_high * 8 bytes of traffic; launch latency dominates).
__global__ void gather_bias_kernel(const float* __restrict__ b, int64_t V,
                                   const int32_t* __restrict__ t2f, int V_high,
                                   float* __restrict__ b_high,
                                   unsigned long long* __restrict__ n_invalid) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < V_high;
       i += gridDim.x * blockDim.x) {
    const int64_t src = t2f[i];
    const bool ok = src >= 0 && src < V;
    b_high[i] = ok ? b[src] : 0.0f;
    if (!ok && n_invalid) atomicAdd(n_invalid, 1ull);
  }
}

}  // namespace
}  // namespace vt

extern "C" vt_status vt_gather_bias(const float* b, int64_t V,
                                    const int32_t* t2f, int32_t V_high,
                                    float* b_high, uint64_t* n_invalid,
                                    void* stream) {
  using namespace vt;
  if (!b || !t2f || !b_high)
    return fail(VT_ERR_INVALID_ARG, "vt_gather_bias: null pointer");
  if (V <= 0 || V_high <= 0)
    return fail(VT_ERR_INVALID_ARG, "vt_gather_bias: need V > 0, V_high > 0");
  if (!aligned(b, 4) || !aligned(b_high, 4))
    return fail(VT_ERR_INVALID_ARG, "vt_gather_bias: b, b_high not 4B aligned");
  if (b < b_high + V_high && b_high < b + V)
    return fail(VT_ERR_INVALID_ARG, "vt_gather_bias: b_high overlaps b");
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  const int grid = (int)std::min<int64_t>(((int64_t)V_high + 255) / 256,
                                          (int64_t)di.num_sms * 4);
  gather_bias_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
      b, V, t2f, V_high, b_high, reinterpret_cast<unsigned long long*>(n_invalid));
  return launch_status("gather_bias_kernel");
}

extern "C" vt_status vt_gather_rows(const uint16_t* W, int64_t V, int32_t d,
                                    const int32_t* t2f, int32_t V_high,
                                    uint16_t* W_high, uint64_t* n_invalid,
                                    void* stream) {
  using namespace vt;
  if (!W || !t2f || !W_high)
    return fail(VT_ERR_INVALID_ARG, "vt_gather_rows: null pointer");
  if (V <= 0 || V_high <= 0 || d <= 0 || d % 8 != 0)
    return fail(VT_ERR_INVALID_ARG,
                "vt_gather_rows: need V > 0, V_high > 0, d > 0, d % 8 == 0");
  if (!aligned(W, 16) || !aligned(W_high, 16))
    return fail(VT_ERR_INVALID_ARG, "vt_gather_rows: W, W_high not 16B aligned");
  const uint16_t* w_end = W + V * (int64_t)d;
  const uint16_t* o_end = W_high + (int64_t)V_high * d;
  if (W < o_end && W_high < w_end)
    return fail(VT_ERR_INVALID_ARG, "vt_gather_rows: W_high overlaps W");
  DeviceInfo di;
  if (!current_device(&di)) return VT_ERR_CUDA;
  const int warps_per_cta = kGatherThreads / 32;
  int64_t want = ((int64_t)V_high + warps_per_cta - 1) / warps_per_cta;
  int grid = (int)std::min<int64_t>(want, (int64_t)di.num_sms * 8);
  gather_rows_kernel<<<grid, kGatherThreads, 0, (cudaStream_t)stream>>>(
      W, V, d, t2f, V_high, W_high,
      reinterpret_cast<unsigned long long*>(n_invalid));
  return launch_status("gather_rows_kernel");
}
