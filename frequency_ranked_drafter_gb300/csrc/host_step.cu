// vt_host_step_* — a draft step from host memory, replayed from a CUDA graph
// owned by the library.
//
// A caller that keeps its hidden states on the host (a CPU-side decode loop,
// a different process's buffers) pays per step for: the copy of the step's
// hidden states to the device, the head, the copy of ids and probabilities
// back, and a synchronise.  The handle captures the three device operations
// once into a CUDA graph on its own stream: a small kernel copies H from a
// pinned staging buffer to the device and lets the head start at once (the
// head is a programmatic dependent: it prefetches its first weight rows
// while H crosses, and waits for the copy before reading it), then
// vt_draft_head_ex, whose last CTA writes ids and probabilities straight into
// a pinned host buffer (pinned memory is addressable from the device, so no
// copy node follows).  A last small kernel, a programmatic dependent of the
// head (its launch overlaps the head), waits for the head to complete,
// moves the head's device error word into the same pinned buffer (clearing
// it), and then, after a system-scope fence, writes the step's sequence
// number there too.  Each step is then a host copy of H into the staging
// buffer, one graph launch, a host wait for that sequence number (a spin on
// the pinned word, which returns ~2.5 us sooner than a stream synchronise;
// a synchronise takes over if the spin runs long, and reports any launch or
// kernel error), a look at the error word and a host copy out.
// The pages have no counterpart: it serves the end-to-end use of the head.
#include <atomic>
#include <cstring>
#include <new>

#include "head_common.cuh"

struct vt_host_step {
  int M, d, k;
  cudaStream_t stream = nullptr;
  cudaGraphExec_t exec = nullptr;
  uint16_t* H_pinned = nullptr;   // host, pinned [M, d]
  int32_t* out_pinned = nullptr;  // host, pinned [2, M, k] (ids, prob bits),
                                  // written by the head's kernel, then the
                                  // head's error word and the step's
                                  // sequence number
  uint16_t* H_dev = nullptr;      // device [M, d]
  void* ws = nullptr;             // device head workspace, then the step
                                  // counter (uint32, after wbytes)
  unsigned seq = 0;               // steps published so far
};

namespace {

constexpr int kCopyThreads = 256;

// dst[i] = src[i] for n 16-byte words, src in pinned host memory.  Triggers
// its dependents first, so the head's grid can become resident meanwhile.
__global__ void __launch_bounds__(kCopyThreads)
    host_h_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                       int n) {
  vt::grid_launch_dependents();
  for (int i = blockIdx.x * kCopyThreads + threadIdx.x; i < n;
       i += gridDim.x * kCopyThreads)
    dst[i] = src[i];
}

// Once the head before it has completed: err_out[0] = *err, *err = 0, then
// the step counter's next value into err_out[1] behind a system-scope
// fence, so a host that reads that value also sees the head's ids and
// probabilities and the error word (err_out in pinned host memory).
__global__ void host_err_publish_kernel(unsigned* err, unsigned* err_out, unsigned* seq) {
  vt::grid_dependency_wait();
  const unsigned e = *err;
  err_out[0] = e;
  if (e) *err = 0u;
  const unsigned n = *seq + 1u;
  *seq = n;
  __threadfence_system();
  *reinterpret_cast<volatile unsigned*>(err_out + 1) = n;
}

// Host spins on the step's sequence number before a synchronise takes over
// (about 10-50 ms of polling).
constexpr long kSpinLimit = 20000000L;

void destroy(vt_host_step* h) {
  if (!h) return;
  if (h->exec) cudaGraphExecDestroy(h->exec);
  if (h->stream) cudaStreamDestroy(h->stream);
  if (h->H_pinned) cudaFreeHost(h->H_pinned);
  if (h->out_pinned) cudaFreeHost(h->out_pinned);
  if (h->H_dev) cudaFree(h->H_dev);
  if (h->ws) cudaFree(h->ws);
  delete h;
}

}  // namespace

extern "C" vt_status vt_host_step_create(const uint16_t* W_high, int32_t V_high,
                                         int32_t d, const int32_t* t2f,
                                         int32_t M, int32_t k,
                                         const vt_head_options* opts,
                                         vt_host_step** out) {
  using namespace vt;
  if (!out) return fail(VT_ERR_INVALID_ARG, "vt_host_step_create: null handle");
  *out = nullptr;
  if (opts && opts->mode == VT_HEAD_SAMPLE)
    return fail(VT_ERR_INVALID_ARG,
                "vt_host_step_create: drawing needs a new step counter per call; "
                "a replayed graph would repeat it");
  if (!W_high || M < 1 || M > 256 || d < 8 || d % 8 || k < 1 || k > kTopKMax ||
      V_high < k)
    return fail(VT_ERR_INVALID_ARG, "vt_host_step_create: bad arguments");
  vt_host_step* h = new (std::nothrow) vt_host_step;
  if (!h) return fail(VT_ERR_CUDA, "vt_host_step_create: out of host memory");
  h->M = M;
  h->d = d;
  h->k = k;
  const size_t hbytes = (size_t)M * d * 2, obytes = (size_t)M * k * 8 + 8;
  const size_t wbytes = vt_draft_head_workspace_size(M, V_high, k);
  auto bad = [&](const char* what) {
    const cudaError_t e = cudaGetLastError();
    destroy(h);
    return fail(VT_ERR_CUDA, std::string("vt_host_step_create: ") + what + ": " +
                                 cudaGetErrorString(e));
  };
  if (cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking) != cudaSuccess)
    return bad("stream");
  if (cudaMallocHost(&h->H_pinned, hbytes) != cudaSuccess ||
      cudaMallocHost(&h->out_pinned, obytes) != cudaSuccess ||
      cudaMalloc(&h->H_dev, hbytes) != cudaSuccess ||
      cudaMalloc(&h->ws, wbytes + 256) != cudaSuccess)
    return bad("allocation");
  std::memset(h->H_pinned, 0, hbytes);
  std::memset(h->out_pinned, 0, obytes);
  if (cudaMemsetAsync(h->ws, 0, wbytes + 256, h->stream) != cudaSuccess) return bad("memset");
  unsigned* seq_dev = reinterpret_cast<unsigned*>(static_cast<char*>(h->ws) + wbytes);
  // the device address of the pinned output buffer (the same pointer under
  // unified addressing)
  int32_t* out_devp = nullptr;
  if (cudaHostGetDevicePointer((void**)&out_devp, h->out_pinned, 0) != cudaSuccess)
    return bad("output buffer mapping");
  int32_t* ids_dev = out_devp;
  float* probs_dev = reinterpret_cast<float*>(out_devp + (size_t)M * k);
  unsigned* err_out = reinterpret_cast<unsigned*>(out_devp + (size_t)2 * M * k);
  unsigned* err_dev = reinterpret_cast<unsigned*>(static_cast<char*>(h->ws) + 128);
  uint16_t* H_src = nullptr;
  if (cudaHostGetDevicePointer((void**)&H_src, h->H_pinned, 0) != cudaSuccess)
    return bad("staging buffer mapping");
  const int n16 = (int)(hbytes / 16);  // d % 8 == 0: whole 16-byte words
  const int copy_blocks = std::min(64, (n16 + kCopyThreads - 1) / kCopyThreads);
  // one eager step first (kernel attributes, first-call set-up), then capture
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1 &&
        cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return bad("begin capture");
    host_h_copy_kernel<<<copy_blocks, kCopyThreads, 0, h->stream>>>(
        reinterpret_cast<const uint4*>(H_src), reinterpret_cast<uint4*>(h->H_dev), n16);
    if (cudaGetLastError() != cudaSuccess) return bad("copy in");
    vt_status st = vt_draft_head_ex(h->H_dev, M, d, d, W_high, V_high, t2f, k,
                                    opts, ids_dev, probs_dev, nullptr, h->ws,
                                    wbytes, h->stream);
    if (st == VT_OK) {
      const cudaError_t pe = launch_dependent(host_err_publish_kernel, dim3(1),
                                              dim3(1), 0, h->stream, err_dev,
                                              err_out, seq_dev);
      if (pe != cudaSuccess) {
        cudaGetLastError();
        st = fail(VT_ERR_CUDA, std::string("host_err_publish_kernel: ") +
                                   cudaGetErrorString(pe));
      }
    }
    if (st != VT_OK) {
      if (pass == 1) {
        cudaGraph_t g = nullptr;
        cudaStreamEndCapture(h->stream, &g);
        if (g) cudaGraphDestroy(g);
      }
      destroy(h);
      return st;
    }
    if (pass == 0) {
      if (cudaStreamSynchronize(h->stream) != cudaSuccess) return bad("first step");
      h->seq = 1;  // the eager step published 1
    }
  }
  cudaGraph_t graph = nullptr;
  if (cudaStreamEndCapture(h->stream, &graph) != cudaSuccess || !graph)
    return bad("end capture");
  const cudaError_t ie = cudaGraphInstantiate(&h->exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ie != cudaSuccess) return bad("instantiate");
  *out = h;
  return VT_OK;
}

extern "C" vt_status vt_host_step_run(vt_host_step* h, const uint16_t* H_host,
                                      int32_t* ids_host, float* probs_host) {
  using namespace vt;
  if (!h || !H_host || !ids_host || !probs_host)
    return fail(VT_ERR_INVALID_ARG, "vt_host_step_run: null pointer");
  const size_t mk = (size_t)h->M * h->k;
  if (H_host != h->H_pinned)
    std::memcpy(h->H_pinned, H_host, (size_t)h->M * h->d * 2);
  if (cudaGraphLaunch(h->exec, h->stream) != cudaSuccess)
    return fail(VT_ERR_CUDA, std::string("vt_host_step_run: ") +
                                 cudaGetErrorString(cudaGetLastError()));
  const unsigned want = ++h->seq;
  volatile unsigned* published = reinterpret_cast<volatile unsigned*>(h->out_pinned + 2 * mk + 1);
  for (long spins = 0; *published != want;) {
    if (++spins > kSpinLimit) {
      // a long step (a busy GPU) or a failed one: wait for the stream
      if (cudaStreamSynchronize(h->stream) != cudaSuccess)
        return fail(VT_ERR_CUDA, std::string("vt_host_step_run: ") +
                                     cudaGetErrorString(cudaGetLastError()));
      if (*published != want)
        return fail(VT_ERR_CUDA, "vt_host_step_run: the step did not publish its result");
      break;
    }
  }
  std::atomic_thread_fence(std::memory_order_acquire);
  const unsigned err = reinterpret_cast<volatile unsigned*>(h->out_pinned)[2 * mk];
  if (err != 0)
    return fail(VT_ERR_TIMEOUT,
                "vt_host_step_run: a bounded wait inside the head gave up; "
                "the step's outputs are incomplete");
  std::memcpy(ids_host, h->out_pinned, mk * 4);
  std::memcpy(probs_host, h->out_pinned + mk, mk * 4);
  return VT_OK;
}

extern "C" uint16_t* vt_host_step_staging(vt_host_step* h) {
  return h ? h->H_pinned : nullptr;
}

extern "C" uint32_t* vt_host_step_error_word(vt_host_step* h) {
  return h ? reinterpret_cast<uint32_t*>(static_cast<char*>(h->ws) + 128) : nullptr;
}

extern "C" void vt_host_step_destroy(vt_host_step* h) {
  if (h) cudaStreamSynchronize(h->stream);
  destroy(h);
}
