// vt_selftest_wait_timeout — makes the library's bounded device wait run
// out, so that a caller (or a test) can see the failure path work: the
// kernel sets the error word and returns, and the context stays usable.
//
// Every wait of the library's kernels on an mbarrier (TMA stages, MMA
// completion, the accumulator hand-over, the final merge's bulk copy) is
// tc::mbar_wait with a cycle budget; on expiry the kernel records
// VT_ERR_TIMEOUT in the workspace error word and stops.  Here one CTA
// initialises an mbarrier on which nothing ever arrives and waits on it with
// the caller's budget.  vt_selftest_check does the same for the debug
// build's bounds checks.  The pages have no counterpart.
#include "head_common.cuh"

namespace vt {
namespace {

__global__ void __launch_bounds__(32)
    wait_timeout_kernel(unsigned* err, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  __syncwarp();
  // nothing arrives on `bar`: the wait gives up after `budget` cycles
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0u, budget))
    atomicExch(err, (unsigned)VT_ERR_TIMEOUT);
}

// buf[i] = i for i = 0 .. n, each write guarded by a check that allows
// only i < n: every write lands inside buf (n + 1 values) in either build,
// and in a bounds-checked build the last one is skipped and reported.
__global__ void check_selftest_kernel(uint32_t* buf, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= n;
       i += gridDim.x * blockDim.x)
    if (VT_CHECKED(i < n)) buf[i] = (uint32_t)i;
}

}  // namespace
}  // namespace vt

extern "C" vt_status vt_selftest_check(uint32_t* buf, int32_t n, void* stream) {
  using namespace vt;
  if (!buf || !aligned(buf, 4) || n < 1 || n > (1 << 30))
    return fail(VT_ERR_INVALID_ARG, "vt_selftest_check: need buf and 1 <= n <= 2^30");
  const int blocks = (int)std::min<int64_t>(((int64_t)n + 256) / 256, 1024);
  check_selftest_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(buf, n);
  return launch_status("check_selftest_kernel");
}

extern "C" vt_status vt_selftest_wait_timeout(uint32_t* err_word,
                                              int64_t budget_cycles,
                                              void* stream) {
  using namespace vt;
  if (!err_word || !aligned(err_word, 4))
    return fail(VT_ERR_INVALID_ARG, "vt_selftest_wait_timeout: null or misaligned error word");
  if (budget_cycles < 1 || budget_cycles > (int64_t(1) << 31))
    return fail(VT_ERR_INVALID_ARG,
                "vt_selftest_wait_timeout: budget must be 1 .. 2^31 cycles");
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err_word, (long long)budget_cycles);
  return launch_status("wait_timeout_kernel");
}
