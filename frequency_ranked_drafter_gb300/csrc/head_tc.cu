// vt_draft_head, tree-draft path (M >= 5 hidden states): a tcgen05 GEMM for
// the logits of all M rows at once, then a per-row softmax + top-k kernel.
//
// "FR-Spec: Accelerating Large-Vocabulary Language Models via
// Frequency-Ranked Speculative Sampling", Method > Key design: the draft
// lm_head projects onto the V_high most frequent tokens only (the pages'
// drafter, EAGLE-2, expands a draft tree, so one step scores many tree
// nodes); "VocabTrim: ...", Implementation Step 4: softmax over the trimmed
// logits, then trimmed index -> full id through trimmed_to_full.
//
// GEMM: logits[m][i] = sum_j H[m][j] * W_high[i][j].  The tensor cores see
// the W_high tile as the MMA's M side (128 rows) and the hidden states as
// its N side (N = M rounded up to 16, at most 256), both K-major, so one
// pass over W_high serves every hidden state.  Per CTA (persistent over
// tiles of 128 rows): warp 0 streams K blocks of 64 (128 bytes, 128-byte
// swizzle) of the W tile and of H into a ring of shared-memory stages with
// TMA; one thread of warp 1 issues tcgen05.mma into a double-buffered TMEM
// accumulator; warps 2-5 read finished accumulators out of TMEM and store
// fp32 logits (tile rows along lanes, so every store is a coalesced 128-byte
// row segment).  At these M the work stays bound by the W_high stream.
//
// Softmax + top-k: one CTA per hidden state reads its V_high logits twice
// from L2: the first pass builds the online (max, sum of exp) and each
// thread's best entry; a warp tournament over those bests gives a lower
// bound on the k-th best logit (a warp's k-th best thread-best has k
// entries at least as good); the second pass keeps only entries reaching
// that bound, which are ranked exactly by counting.
//
// Every wait on an mbarrier is bounded (kWaitBudget cycles, about a
// second); a wait that gives up records VT_ERR_TIMEOUT in the error word of
// the workspace, the CTA stops issuing work, drains what it issued and
// frees its TMEM before returning.
#include <cudaTypedefs.h>

#include <mutex>

#include "head_common.cuh"
#include "tc_ptx.cuh"

namespace vt {
namespace {

constexpr int kTcThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr int kTcMaxStages = 6;
constexpr int kTcBlockK = 64;  // bf16 per K block: 128 bytes, one swizzle row
constexpr int kTcTileRows = 128;
constexpr int kTcABytes = kTcTileRows * kTcBlockK * 2;  // 16 KB
constexpr long long kWaitBudget = 2000000000LL;

struct TcArgs {
  int V_high, d, M, N, NB;  // NB: TMEM column stride of one accumulator
  int stages;
  uint32_t tmem_cols;
  float* logits;  // [M][V_high]
  unsigned* err;
};

__device__ __forceinline__ void record_error(unsigned* err, volatile int* abort) {
  *abort = 1;
  atomicExch(err, (unsigned)VT_ERR_TIMEOUT);
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > kWaitBudget) return false;
  }
  return true;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    head_tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmH, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kTcMaxStages], empty[kTcMaxStages];
  __shared__ __align__(8) uint64_t tfull[2], tempty[2], drain;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;
  const int b_bytes = a.N * kTcBlockK * 2;
  const int stage_bytes = kTcABytes + b_bytes;
  const int ntiles = (a.V_high + kTcTileRows - 1) / kTcTileRows;
  const int nkb = (a.d + kTcBlockK - 1) / kTcBlockK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 4);
    }
    tc::mbar_init(&drain, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, a.tmem_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------- TMA producer
      tc::prefetch_tensormap(&tmW);
      tc::prefetch_tensormap(&tmH);
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;  // loads issued, for the drain on abort
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_or_abort(&empty[s], ph ^ 1u, &abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + (size_t)s * stage_bytes;
          tc::mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
          tc::tma_load_2d(st, &tmW, &full[s], kb * kTcBlockK, tile * kTcTileRows);
          tc::tma_load_2d(st + kTcABytes, &tmH, &full[s], kb * kTcBlockK, 0);
          ++issued;
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        record_error(a.err, &abort_flag);
        // drain: the last min(issued, S) stages may still be landing
        const int n = issued < S ? issued : S;
        int ds = s, dph = ph;
        for (int i = 0; i < n; ++i) {
          if (--ds < 0) { ds = S - 1; dph ^= 1u; }
          tc::mbar_wait(&full[ds], dph, kWaitBudget);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------- MMA issuer
      const uint32_t idesc = tc::idesc_bf16_f32(kTcTileRows, a.N);
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!wait_or_abort(&tempty[acc], aph ^ 1u, &abort_flag)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * a.NB);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_or_abort(&full[s], ph, &abort_flag)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t a_base = tc::smem_u32(smem + (size_t)s * stage_bytes);
          const uint32_t b_base = a_base + kTcABytes;
#pragma unroll
          for (int j = 0; j < kTcBlockK / 16; ++j)
            tc::mma_bf16(d_tmem, tc::sdesc_k_sw128(a_base + 32 * j),
                         tc::sdesc_k_sw128(b_base + 32 * j), idesc,
                         (kb > 0 || j > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);  // stage reusable once these complete
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc::mma_commit(&tfull[acc]);
      }
      if (!ok) {
        record_error(a.err, &abort_flag);
        // let every MMA issued so far finish before TMEM is released
        tc::mma_commit(&drain);
        tc::mbar_wait(&drain, 0u, kWaitBudget);
      }
    }
  } else {  // --------------------------------------------- epilogue warps
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int it = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      if (!wait_or_abort(&tfull[acc], aph, &abort_flag)) {
        if (lane == 0) record_error(a.err, &abort_flag);
        break;
      }
      tc::tc_fence_after();
      const int row = tile * kTcTileRows + 32 * q + lane;
      for (int c0 = 0; c0 < a.N; c0 += 32) {
        float r[32];
        tc::tmem_ld_32x32(tmem + ((uint32_t)(32 * q) << 16) +
                              (uint32_t)(acc * a.NB + c0),
                          r);
        tc::tmem_ld_wait();
        if (row < a.V_high) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < a.M) a.logits[(size_t)(c0 + j) * a.V_high + row] = r[j];
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[acc]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, a.tmem_cols);
  }
}

// ------------------------------------------------- per-row softmax + top-k
constexpr int kRowThreads = 512;
constexpr int kRowSurvivors = 4096;

__global__ void __launch_bounds__(kRowThreads)
    rows_topk_kernel(const float* __restrict__ logits, int V_high, int k,
                     const int32_t* __restrict__ t2f,
                     int32_t* __restrict__ out_ids,
                     float* __restrict__ out_probs) {
  constexpr int kWarps = kRowThreads / 32;
  __shared__ float red[kWarps];
  __shared__ float tw_v[kWarps];
  __shared__ int tw_i[kWarps];
  __shared__ float2 surv[kRowSurvivors];
  __shared__ int s_cnt;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = logits + (size_t)blockIdx.x * V_high;
  int32_t* ids = out_ids + (size_t)blockIdx.x * k;
  float* probs = out_probs + (size_t)blockIdx.x * k;

  // pass 1: online (max, sumexp) and this thread's best entry
  float mx = -INFINITY, se = 0.f, bv = -INFINITY;
  int bi = INT_MAX;
  for (int i = tid; i < V_high; i += kRowThreads) {
    const float v = __ldcg(row + i);
    if (v > mx) { se = se * __expf(mx - v) + 1.f; mx = v; }
    else se += __expf(v - mx);
    if (v > bv) { bv = v; bi = i; }  // i grows: the first of equals stays
  }
  if (tid == 0) s_cnt = 0;
  const float mg = block_max<kRowThreads>(mx, red);
  const float sg = block_sum<kRowThreads>(se > 0.f ? se * __expf(mx - mg) : 0.f, red);

  // lower bound on the k-th best: per warp, the k-th best thread-best
  {
    float tv = -INFINITY;
    int ti = INT_MAX;
    float lv = bv;
    int li = bi;
    for (int r = 0; r < k; ++r) {
      const unsigned lk = li != INT_MAX ? float_key(lv) : 0u;
      const unsigned wk = __reduce_max_sync(~0u, lk);
      if (wk == 0u) { tv = -INFINITY; ti = INT_MAX; break; }  // fewer than k
      const int wi = (int)__reduce_min_sync(~0u, lk == wk ? (unsigned)li : 0xffffffffu);
      const unsigned owner = __ballot_sync(~0u, lk == wk && li == wi);
      const float wv = __shfl_sync(~0u, lv, __ffs(owner) - 1);
      tv = wv;
      ti = wi;
      if (lk == wk && li == wi) { lv = -INFINITY; li = INT_MAX; }
    }
    if (lane == 0) { tw_v[warp] = tv; tw_i[warp] = ti; }
  }
  __syncthreads();
  float T_v = tw_v[0];
  int T_i = tw_i[0];
  for (int w = 1; w < kWarps; ++w)
    if (tw_i[w] != INT_MAX && key_beats(tw_v[w], tw_i[w], T_v, T_i)) {
      T_v = tw_v[w]; T_i = tw_i[w];
    }

  // pass 2: entries not beaten by the bound
  for (int i = tid; i < V_high; i += kRowThreads) {
    const float v = __ldcg(row + i);
    if (!key_beats(T_v, T_i, v, i)) {
      const int p = atomicAdd(&s_cnt, 1);
      if (p < kRowSurvivors) surv[p] = make_float2(v, __int_as_float(i));
    }
  }
  __syncthreads();
  const int S = s_cnt;
  if (S <= kRowSurvivors) {
    for (int c = tid; c < S; c += kRowThreads) {
      const float v = surv[c].x;
      const int i = __float_as_int(surv[c].y);
      int rank = 0;
      for (int q = 0; q < S; ++q)
        rank += key_beats(surv[q].x, __float_as_int(surv[q].y), v, i);
      if (rank < k) {
        ids[rank] = t2f ? t2f[i] : i;
        probs[rank] = expf(v - mg) / sg;
      }
    }
  } else {  // more survivors than the buffer (pathological): k arg-max rounds
    float pv = INFINITY;
    int pi = INT_MIN;
    for (int r = 0; r < k; ++r) {
      float bv2 = -INFINITY;
      int bi2 = INT_MAX;
      for (int i = tid; i < V_high; i += kRowThreads) {
        const float v = __ldcg(row + i);
        if (key_beats(pv, pi, v, i) && key_beats(v, i, bv2, bi2)) { bv2 = v; bi2 = i; }
      }
      block_best<kRowThreads>(bv2, bi2, tw_v, tw_i);
      if (tid == 0) {
        ids[r] = bi2 == INT_MAX ? -1 : (t2f ? t2f[bi2] : bi2);
        probs[r] = bi2 == INT_MAX ? 0.f : expf(bv2 - mg) / sg;
      }
      pv = bv2;
      pi = bi2;
    }
  }
}

// ------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map: rows x cols (cols contiguous, row pitch ld elements),
// box of 64 columns (128 bytes) x box_rows, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
              uint64_t ld, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTcBlockK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t head_tc_workspace(int M, int V_high) {
  return 256 + (size_t)M * V_high * sizeof(float);
}

vt_status head_tc(const uint16_t* H, int M, int d, int64_t ldh,
                  const uint16_t* W, int V_high, const int32_t* t2f, int k,
                  int32_t* out_ids, float* out_probs, float* out_logits,
                  void* ws, const DeviceInfo& di, cudaStream_t s) {
  if (M > 256) return fail(VT_ERR_UNSUPPORTED, "head_tc: M > 256");
  unsigned* err = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 128);
  float* logits = out_logits ? out_logits
                             : reinterpret_cast<float*>(static_cast<char*>(ws) + 256);
  TcArgs a;
  a.V_high = V_high;
  a.d = d;
  a.M = M;
  a.N = (M + 15) / 16 * 16;
  a.NB = (a.N + 31) / 32 * 32;
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * a.NB)) cols <<= 1;
  a.tmem_cols = cols;
  a.logits = logits;
  a.err = err;
  const int stage_bytes = kTcABytes + a.N * kTcBlockK * 2;
  a.stages = std::min<int>(kTcMaxStages, (di.max_smem_optin - 4096) / stage_bytes);
  if (a.stages < 2) return fail(VT_ERR_UNSUPPORTED, "head_tc: stages do not fit");
  CUtensorMap tmW, tmH;
  if (!make_map(&tmW, W, (uint64_t)V_high, (uint64_t)d, (uint64_t)d, kTcTileRows) ||
      !make_map(&tmH, H, (uint64_t)M, (uint64_t)d, (uint64_t)ldh, (uint32_t)a.N))
    return fail(VT_ERR_CUDA, "head_tc: cuTensorMapEncodeTiled failed");
  if (!allow_max_smem(head_tc_gemm_kernel, di)) return VT_ERR_CUDA;
  const int ntiles = (V_high + kTcTileRows - 1) / kTcTileRows;
  const int grid = std::min(ntiles, di.num_sms);
  const int smem = a.stages * stage_bytes + 1024;
  head_tc_gemm_kernel<<<grid, kTcThreads, smem, s>>>(tmW, tmH, a);
  vt_status st = launch_status("head_tc_gemm_kernel");
  if (st != VT_OK) return st;
  rows_topk_kernel<<<M, kRowThreads, 0, s>>>(logits, V_high, k, t2f, out_ids,
                                             out_probs);
  return launch_status("rows_topk_kernel");
}

}  // namespace vt
