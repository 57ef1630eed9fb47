// vt_draft_head, tree-draft path (M >= 2 hidden states): a tcgen05 GEMM for
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
// TMA (a stage is up to four such K blocks of the same rows, requested back
// to back); one thread of warp 1 issues tcgen05.mma into a double-buffered TMEM
// accumulator; warps 2-17 read finished accumulators out of TMEM (four warps
// per 32-lane quadrant, each every fourth 16-column chunk, so the last
// tile's epilogue, which nothing overlaps, is spread over all sixteen) and
// store fp32 logits (tile rows along lanes, so every store is a coalesced
// 128-byte row segment).  At these M the work stays bound by the W_high
// stream.
//
// Softmax + top-k: each hidden state's V_high logits (L2-resident, bias
// added by the GEMM epilogue) are split over CTAs of 4096; each CTA reduces
// its part to (max, sum of exp of logit/T, exact top-k of the selection
// score) and the last CTA of the row merges the parts.  The score is
// logit/T, or logit/T plus the token's Gumbel noise when sampling.  Entries
// carry their full-vocabulary id (t2f read next to the logits), which breaks
// ties between equal scores (lower id first) and is what the call returns.
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

// warp 0 TMA, warp 1 MMA + TMEM, warps 2-17 epilogue (four warps per TMEM
// lane quadrant, each taking every fourth 16-column chunk of the
// accumulator).  The last tile's epilogue is exposed: with 8 warps and
// 32-column chunks it took ~2 us at N = 64, most of it the quadrant
// statistics' shuffles and exponentials of one chunk per warp.
constexpr int kTcThreads = 576;
constexpr int kTcEpilogueWarps = 16;
constexpr int kTcChunk = 16;  // accumulator columns (hidden states) per chunk
constexpr int kTcMaxStages = 6;
// k-blocks of a CTA's first W_high tile prefetched into L2 before the
// dependency wait.
constexpr int kTcPrefetchKBlocks = 32;
constexpr int kTcBlockK = 64;  // bf16 per K atom: 128 bytes, one swizzle row
// A stage holds up to kTcMaxAtoms K atoms (adjacent 128-byte pieces of the
// same 128 W_high rows, loaded back to back), as many as leave kTcMinStages
// stages: wider stages keep more of W_high in flight per SM (M = 60,
// V_high = 32768: 68.5 us with one atom a stage, 59.2 us with two, 53.0
// with three).
constexpr int kTcMaxAtoms = 4;
constexpr int kTcMinStages = 3;
constexpr int kTcTileRows = 128;
constexpr int kTcABytes = kTcTileRows * kTcBlockK * 2;  // 16 KB
constexpr long long kWaitBudget = 2000000000LL;

struct TcArgs {
  int V_high, d, M, N, NB;  // NB: TMEM column stride of one accumulator
  int stages;
  int atoms;  // K atoms (64 columns, 128 bytes a row) per stage
  uint32_t tmem_cols;
  float* logits;  // [M][V_high]
  const float* bias;  // [V_high] or null, added to every logit
  unsigned* err;
  // top-k calls: per hidden state m and 32-row quadrant q of the tiles,
  // (max, sum of exp(s - max)) of s = logit / T, at qstat[m * nq + q]
  float2* qstat;
  int nq;
  float inv_tau;
  // 0: each CTA takes whole tiles (tile = blockIdx.x, blockIdx.x + grid, ...).
  // 1: clusters of two CTAs per tile, rank r summing K stages
  // [r * nkb / 2, (r + 1) * nkb / 2); each CTA sends the partner its partial
  // sums of the partner's half of the rows through distributed shared memory
  // and finishes its own half (rank 0 rows 0-63, rank 1 rows 64-127).
  int ksplit;
};

// ------------------------------------------------ thread-block clusters
// This CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives and waits (release /
// acquire at cluster scope): shared-memory set-up before it is visible to
// the other CTAs, and no CTA leaves while another may still access its
// shared memory.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address, in the cluster's shared window, of this CTA's shared
// variable at `smem_addr` as seen in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr), "r"(rank));
  return d;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster, releasing this
// thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}

// try_wait with acquire at cluster scope (the arrivals came from another CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(tc::smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}



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

// Merges two (max, sum of exp(x - max)) pairs of the same hidden state:
// (m1, s1) + (m2, s2) = (max, s_max + s_min * exp(min - max)), where s_max
// belongs to the pair with the larger max.  An empty pair (-inf, 0) adds
// nothing.
__device__ __forceinline__ void merge_stat(float& m, float& s, float pm, float ps) {
  const float hi = fmaxf(m, pm), lo = fminf(m, pm);
  const float e = lo > -INFINITY ? __expf(lo - hi) : 0.f;
  s = m >= pm ? fmaf(ps, e, s) : fmaf(s, e, ps);
  m = hi;
}

// Softmax statistics of one 32-row quadrant of a tile for the chunk's
// hidden states c0 .. c0+15: max of s = logit / T over the quadrant's rows
// (rows past V_high excluded) and the sum of exp(s - max).  Each lane
// starts from its row's pairs (s, 1); the pairs are merged across lanes
// along a transposed halving (at each step a lane keeps half of its hidden
// states and merges its partner's pairs for that half, one shuffle pair and
// one exponential per merge), so after four steps lane l holds hidden state
// c0 + (l & 15) over its half-warp, and one more merge with lane l ^ 16
// covers all 32 rows; lanes 0-15 write the pairs.  The row kernel folds
// these into the softmax normaliser and bounds the k-th best score from
// them.
__device__ __forceinline__ void quadrant_stats(const TcArgs& a, const float (&r)[kTcChunk],
                                               int row, int c0, int quad) {
  const int lane = threadIdx.x & 31;
  const bool valid = row < a.V_high;
  float m[kTcChunk], sm[kTcChunk];
#pragma unroll
  for (int j = 0; j < kTcChunk; ++j) {
    m[j] = valid ? __fmul_rn(r[j], a.inv_tau) : -INFINITY;
    sm[j] = valid ? 1.f : 0.f;
  }
#pragma unroll
  for (int h = kTcChunk / 2; h >= 1; h >>= 1) {
    const bool up = (lane & h) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      float km = up ? m[i + h] : m[i], ks = up ? sm[i + h] : sm[i];
      const float om = up ? m[i] : m[i + h], os = up ? sm[i] : sm[i + h];
      merge_stat(km, ks, __shfl_xor_sync(~0u, om, h), __shfl_xor_sync(~0u, os, h));
      m[i] = km;
      sm[i] = ks;
    }
  }
  merge_stat(m[0], sm[0], __shfl_xor_sync(~0u, m[0], 16), __shfl_xor_sync(~0u, sm[0], 16));
  if (lane < kTcChunk && c0 + lane < a.M && VT_CHECKED(quad < a.nq))
    a.qstat[(size_t)(c0 + lane) * a.nq + quad] = make_float2(m[0], sm[0]);
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
  const int b_bytes = a.N * kTcBlockK * 2;  // one K atom of H
  const int A = a.atoms;
  const int stage_bytes = A * (kTcABytes + b_bytes);
  const int ntiles = (a.V_high + kTcTileRows - 1) / kTcTileRows;
  const int natoms = (a.d + kTcBlockK - 1) / kTcBlockK;  // K atoms in all
  const int nkb = (natoms + A - 1) / A;                   // stages per tile
  // this CTA's tiles and K stages
  const uint32_t rank = a.ksplit ? cluster_rank() : 0u;
  const int tile0 = a.ksplit ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int tstep = a.ksplit ? ntiles : (int)gridDim.x;
  const int kb_lo = a.ksplit ? (int)rank * nkb / 2 : 0;
  const int kb_hi = a.ksplit ? ((int)rank + 1) * nkb / 2 : nkb;
  // K split: the partner's partial sums of this CTA's rows land in xbuf,
  // [N][64] fp32 after the stages, and xfull completes when all 256 of the
  // partner's sending threads have arrived
  __shared__ __align__(8) uint64_t xfull;
  float* xbuf = reinterpret_cast<float*>(smem + (size_t)S * stage_bytes);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], kTcEpilogueWarps);
    }
    tc::mbar_init(&drain, 1);
    tc::mbar_init(&xfull, 32 * kTcEpilogueWarps / 2);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, a.tmem_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (a.ksplit) cluster_sync();  // the partner's xfull exists before any arrival
  const uint32_t tmem = tmem_base;
  // the per-row kernel (a programmatic dependent) may become resident now;
  // it waits for this grid's completion before reading the logits
  grid_launch_dependents();
  // This grid is itself a programmatic dependent of the work ahead of it
  // (the previous draft step's row kernel, or the layer that wrote H): until
  // that ends, the producer only asks L2 for the first k-blocks of this
  // CTA's first W_high tile (weights; the TMA loads that use them come after
  // the wait).  Nothing else is read, and no logit written, before it.
  if (warp == 0 && lane == 0 && tile0 < ntiles) {
    tc::prefetch_tensormap(&tmW);
    tc::prefetch_tensormap(&tmH);
    const int x1 = min(min(natoms, kb_hi * A), kb_lo * A + kTcPrefetchKBlocks);
    for (int x = kb_lo * A; x < x1; ++x)
      tc::tma_prefetch_l2_2d(&tmW, x * kTcBlockK, tile0 * kTcTileRows);
  }
  grid_dependency_wait();

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------- TMA producer
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;  // loads issued, for the drain on abort
      bool ok = true;
      for (int tile = tile0; ok && tile < ntiles; tile += tstep) {
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!wait_or_abort(&empty[s], ph ^ 1u, &abort_flag)) {
            ok = false;
            break;
          }
          // the stage's K atoms of the W tile are adjacent 128-byte pieces
          // of the same rows, requested back to back; then H's
          uint8_t* st = smem + (size_t)s * stage_bytes;
          const int na = min(A, natoms - kb * A);
          tc::mbar_arrive_expect_tx(&full[s], (uint32_t)(na * (kTcABytes + b_bytes)));
          for (int x = 0; x < na; ++x)
            tc::tma_load_2d(st + x * kTcABytes, &tmW, &full[s],
                            (kb * A + x) * kTcBlockK, tile * kTcTileRows);
          for (int x = 0; x < na; ++x)
            tc::tma_load_2d(st + A * kTcABytes + x * b_bytes, &tmH, &full[s],
                            (kb * A + x) * kTcBlockK, 0);
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
      for (int tile = tile0; ok && tile < ntiles; tile += tstep, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!wait_or_abort(&tempty[acc], aph ^ 1u, &abort_flag)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * a.NB);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!wait_or_abort(&full[s], ph, &abort_flag)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t a_base = tc::smem_u32(smem + (size_t)s * stage_bytes);
          const uint32_t b_base = a_base + A * kTcABytes;
          const int na = min(A, natoms - kb * A);
          for (int x = 0; x < na; ++x)
#pragma unroll
            for (int j = 0; j < kTcBlockK / 16; ++j)
              tc::mma_bf16(d_tmem,
                           tc::sdesc_k_sw128(a_base + x * kTcABytes + 32 * j),
                           tc::sdesc_k_sw128(b_base + x * b_bytes + 32 * j), idesc,
                           (kb > kb_lo || x > 0 || j > 0) ? 1u : 0u);
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
    const int part = (warp - 2) >> 2;  // which chunks of the accumulator
    // K split: the partner finishes the rows of this warp's quadrant (send)
    // or this CTA does and adds the partner's part (receive)
    const bool send = a.ksplit && (uint32_t)(q >> 1) != rank;
    const bool recv = a.ksplit && !send;
    const int xrow = 32 * (q & 1) + lane;  // the row within a CTA's half
    int it = 0;
    for (int tile = tile0; tile < ntiles; tile += tstep, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      if (!wait_or_abort(&tfull[acc], aph, &abort_flag)) {
        if (lane == 0) record_error(a.err, &abort_flag);
        break;
      }
      tc::tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * a.NB);
      if (send) {
        const uint32_t xb = map_to_rank(tc::smem_u32(xbuf), rank ^ 1u);
        for (int c0 = kTcChunk * part; c0 < a.N; c0 += 4 * kTcChunk) {
          float r[kTcChunk];
          tc::tmem_ld_32x32_x16(tacc + (uint32_t)c0, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < kTcChunk; ++j)
            if (c0 + j < a.M) st_cluster_f32(xb + (uint32_t)(((c0 + j) * 64 + xrow) * 4), r[j]);
        }
        mbar_arrive_cluster(map_to_rank(tc::smem_u32(&xfull), rank ^ 1u));
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty[acc]);
        continue;
      }
      if (recv) {  // the partner's part of these rows (bounded wait)
        bool ok = mbar_try_wait_cluster(&xfull, 0u);
        const long long t0 = clock64();
        while (!ok && !abort_flag && clock64() - t0 <= kWaitBudget)
          ok = mbar_try_wait_cluster(&xfull, 0u);
        if (!ok) {
          if (lane == 0) record_error(a.err, &abort_flag);
          break;
        }
      }
      const int row = tile * kTcTileRows + 32 * q + lane;
      const float b = row < a.V_high && a.bias ? __ldg(a.bias + row) : 0.f;
      for (int c0 = kTcChunk * part; c0 < a.N; c0 += 4 * kTcChunk) {
        float r[kTcChunk];
        tc::tmem_ld_32x32_x16(tacc + (uint32_t)c0, r);
        tc::tmem_ld_wait();
        if (recv) {
#pragma unroll
          for (int j = 0; j < kTcChunk; ++j)
            if (c0 + j < a.M) r[j] += xbuf[(c0 + j) * 64 + xrow];
        }
#pragma unroll
        for (int j = 0; j < kTcChunk; ++j) r[j] += b;
        if (row < a.V_high) {
#pragma unroll
          for (int j = 0; j < kTcChunk; ++j)
            if (c0 + j < a.M) a.logits[(size_t)(c0 + j) * a.V_high + row] = r[j];
        }
        if (a.qstat) quadrant_stats(a, r, row, c0, tile * 4 + q);
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
  // K split: neither CTA leaves while its partner may still write into its
  // shared memory
  if (a.ksplit) cluster_sync();
}

// ------------------------------------------------- per-row softmax + top-k
// Grid: M rows x P parts.  Each CTA owns kRowSpan consecutive logits of one
// row (kRowVals per thread, loaded once into registers with float4 loads),
// computes their (max, sum of exp) and their exact top-k, publishes them as
// a partial, and the last CTA of the row to arrive (ticket per row, acquire
// -release) merges the row's P partials and writes ids and probabilities.
//
// Exact top-k of a CTA's values: each warp's k-th best thread-best (a warp
// tournament with redux.sync) bounds the CTA's k-th best from below (those k
// thread-bests are k values at least that good); only values reaching the
// best such bound are kept, and they are ranked by counting.
constexpr int kRowThreads = 256;
constexpr int kRowVals = 16;
constexpr int kRowSpan = kRowThreads * kRowVals;  // 4096 logits per CTA
// Survivors of one CTA: every value of its span can survive in the worst
// case (a span's values at or above T number at most k per warp's threads
// times kRowVals, which for k = 32 is the whole span), so the buffer holds
// the span.
constexpr int kRowSurvivors = kRowSpan;
constexpr int kRowSmem = kRowSurvivors * (sizeof(float2) + sizeof(float));

struct RowArgs {
  const float* logits;  // [M][V_high], bias already added
  int V_high, k, P;
  const int32_t* t2f;
  int32_t* out_ids;
  float* out_probs;
  unsigned* tickets;  // [M], zero between calls
  float* part;        // [M][P][2 + 3k]
  float inv_tau;  // 1 / T
  int sample;
  uint64_t seed, offset;
  const int32_t* row_ids;  // noise index of each row (null: the row)
};

// Selection score of one logit: s = logit / T, plus the token's Gumbel noise
// when sampling.
__device__ __forceinline__ float row_score(const RowArgs& a, int m, float s, int f) {
  return a.sample ? s + gumbel_noise(a.seed, a.offset, a.row_ids ? __ldg(a.row_ids + m) : m, f)
                  : s;
}

// At most 64 registers a thread, so four CTAs share an SM and a launch of
// up to 4 * SMs CTAs runs in one wave.  Launched as a programmatic
// dependent of the GEMM: its CTAs may be resident early and wait for the
// logits in griddepcontrol.wait.
__global__ void __launch_bounds__(kRowThreads, 4)
    rows_topk_kernel(RowArgs a) {
  constexpr int kWarps = kRowThreads / 32;
  __shared__ float red[kWarps];
  __shared__ float tw_v[kWarps];
  __shared__ int tw_i[kWarps];
  extern __shared__ __align__(16) float2 surv[];  // [kRowSurvivors] (score, full id)
  float* surv_s = reinterpret_cast<float*>(surv + kRowSurvivors);  // logit / T
  __shared__ int s_cnt, s_last;
  grid_dependency_wait();
  // the GEMM has ended: the next draft step's GEMM (a programmatic
  // dependent) may now start its weight prefetch beside this kernel
  grid_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = blockIdx.y, part_idx = blockIdx.x, k = a.k;
  const int ps = 2 + 3 * k;
  const float* row = a.logits + (size_t)m * a.V_high;
  const int base = part_idx * kRowSpan;

  // this thread's values: 4 float4 at base + 4*(tid + 256*q) (or scalars
  // when the row is not 16-byte aligned or at the tail) as s = logit / T,
  // their full-vocabulary ids (which break ties between equal scores) and
  // their selection scores
  float v[kRowVals], sc[kRowVals];
  int f[kRowVals];
  const bool vec = ((a.V_high & 3) == 0) &&
                   ((reinterpret_cast<uintptr_t>(a.logits) & 15) == 0);
#pragma unroll
  for (int q = 0; q < kRowVals / 4; ++q) {
    const int i0 = base + 4 * (tid + kRowThreads * q);
    if (vec && i0 + 3 < a.V_high) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(row + i0));
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        v[4 * q + e] = i0 + e < a.V_high ? __ldcg(row + i0 + e) : -INFINITY;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = i0 + e;
      f[4 * q + e] = i < a.V_high ? (a.t2f ? __ldg(a.t2f + i) : i) : INT_MAX;
    }
  }
  auto idx_of = [&](int j) { return base + 4 * (tid + kRowThreads * (j >> 2)) + (j & 3); };

  float mx = -INFINITY, bv = -INFINITY;
  int bi = INT_MAX;
#pragma unroll
  for (int j = 0; j < kRowVals; ++j) {
    const bool in = idx_of(j) < a.V_high;
    v[j] = in ? v[j] * a.inv_tau : -INFINITY;
    sc[j] = in ? row_score(a, m, v[j], f[j]) : -INFINITY;
    mx = fmaxf(mx, v[j]);
    if (in && key_beats(sc[j], f[j], bv, bi)) { bv = sc[j]; bi = f[j]; }
  }
  float se = 0.f;
  if (mx > -INFINITY) {
#pragma unroll
    for (int j = 0; j < kRowVals; ++j) se += __expf(v[j] - mx);
  }
  if (tid == 0) s_cnt = 0;
  const float cm = block_max<kRowThreads>(mx, red);
  const float cs = block_sum<kRowThreads>(se > 0.f ? se * __expf(mx - cm) : 0.f, red);

  {  // per-warp bound: the k-th best thread-best of the warp
    float tv = -INFINITY;
    int ti = INT_MAX;
    float lv = bv;
    int li = bi;
    for (int r = 0; r < k; ++r) {
      const unsigned lk = li != INT_MAX ? float_key(lv) : 0u;
      const unsigned wk = __reduce_max_sync(~0u, lk);
      if (wk == 0u) { tv = -INFINITY; ti = INT_MAX; break; }
      const int wi = (int)__reduce_min_sync(~0u, lk == wk ? (unsigned)li : 0xffffffffu);
      const unsigned owner = __ballot_sync(~0u, lk == wk && li == wi);
      tv = __shfl_sync(~0u, lv, __ffs(owner) - 1);
      ti = wi;
      if (lk == wk && li == wi) { lv = -INFINITY; li = INT_MAX; }
    }
    if (lane == 0) { tw_v[warp] = tv; tw_i[warp] = ti; }
  }
  __syncthreads();
  float T_v = -INFINITY;
  int T_i = INT_MAX;
  for (int w = 0; w < kWarps; ++w)
    if (tw_i[w] != INT_MAX && key_beats(tw_v[w], tw_i[w], T_v, T_i)) {
      T_v = tw_v[w]; T_i = tw_i[w];
    }
#pragma unroll
  for (int j = 0; j < kRowVals; ++j) {
    if (idx_of(j) < a.V_high && !key_beats(T_v, T_i, sc[j], f[j])) {
      const int p = atomicAdd(&s_cnt, 1);
      if (p < kRowSurvivors) {
        surv[p] = make_float2(sc[j], __int_as_float(f[j]));
        surv_s[p] = v[j];
      }
    }
  }
  __syncthreads();
  float* mypart = a.part + ((size_t)m * a.P + (VT_CHECKED(part_idx < a.P) ? part_idx : 0)) * ps;
  const int S = min(s_cnt, kRowSurvivors);
  // slots this CTA cannot fill stay (-inf, INT_MAX)
  for (int r = tid; r < k; r += kRowThreads) {
    mypart[2 + r] = -INFINITY;
    reinterpret_cast<int*>(mypart)[2 + k + r] = INT_MAX;
    mypart[2 + 2 * k + r] = -INFINITY;
  }
  __syncthreads();
  for (int c = tid; c < S; c += kRowThreads) {
    const float x = surv[c].x;
    const int i = __float_as_int(surv[c].y);
    int rank = 0;
    for (int q = 0; q < S; ++q) rank += key_beats(surv[q].x, __float_as_int(surv[q].y), x, i);
    if (rank < k) {
      mypart[2 + rank] = x;
      reinterpret_cast<int*>(mypart)[2 + k + rank] = i;
      mypart[2 + 2 * k + rank] = surv_s[c];
    }
  }
  if (tid == 0) { mypart[0] = cm; mypart[1] = cs; }

  // ---- last CTA of the row merges the row's P partials
  __syncthreads();
  if (tid == 0) s_last = ticket_arrive(a.tickets + m) == (unsigned)(a.P - 1);
  __syncthreads();
  if (!s_last) return;
  const float* rp = a.part + (size_t)m * a.P * ps;
  float pm = -INFINITY, psum = 0.f;
  for (int b = tid; b < a.P; b += kRowThreads) pm = fmaxf(pm, __ldcg(rp + (size_t)b * ps));
  const float mg = block_max<kRowThreads>(pm, red);
  for (int b = tid; b < a.P; b += kRowThreads) {
    const float s = __ldcg(rp + (size_t)b * ps + 1);
    if (s > 0.f) psum += s * __expf(__ldcg(rp + (size_t)b * ps) - mg);
  }
  const float sg = block_sum<kRowThreads>(psum, red);
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  const int nc = a.P * k;  // all partial candidates (P*k <= kRowSurvivors)
  for (int c = tid; c < nc; c += kRowThreads) {
    const int b = c / k, r = c - b * k;
    const float x = __ldcg(rp + (size_t)b * ps + 2 + r);
    const int i = __ldcg(reinterpret_cast<const int*>(rp + (size_t)b * ps) + 2 + k + r);
    surv[c] = make_float2(x, __int_as_float(i));
    surv_s[c] = __ldcg(rp + (size_t)b * ps + 2 + 2 * k + r);
  }
  __syncthreads();
  int32_t* ids = a.out_ids + (size_t)m * k;
  float* probs = a.out_probs + (size_t)m * k;
  for (int c = tid; c < nc; c += kRowThreads) {
    const float x = surv[c].x;
    const int i = __float_as_int(surv[c].y);
    if (i == INT_MAX) continue;
    int rank = 0;
    for (int q = 0; q < nc; ++q) rank += key_beats(surv[q].x, __float_as_int(surv[q].y), x, i);
    if (rank < k) {
      ids[rank] = i;
      probs[rank] = expf(surv_s[c] - mg) / sg;
    }
  }
  if (tid == 0) a.tickets[m] = 0u;
}

// ------------------------------------------- per-row top-k from statistics
// Top-k calls (no sampling).  One CTA per hidden state m, after the GEMM:
//   * folds the quadrant statistics into the softmax normaliser:
//     Mg = max_q max_q,  Sg = sum_q sum_q * exp(max_q - Mg);
//   * bounds the k-th best score from below: quadrants are dealt into 32
//     disjoint groups by index mod 32 (every group holds some once there
//     are 32 quadrants); the k-th largest of the group maxima is the score
//     of one of k different logits, so it is at most the k-th best score, L;
//   * a logit with s >= L lies in a quadrant whose maximum is >= L: only
//     those quadrants (a few dozen on real data) are read, 32 logits each,
//     and the keys (s, full id) with s >= L are kept in shared memory,
//     ranked by counting, and the k best written as ids and
//     exp(s - Mg) / Sg.
// If more than kSelQuads quadrants reach L, the whole row is scanned
// instead.  If more than kSelCap keys reach L (scores tied at the top), the exact
// k-th best key is found instead by an 8-bit radix select over the 64-bit
// keys (keys are distinct: the full id breaks ties), then the k keys at or
// above it are ranked.
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;  // >= kTopKMax groups
constexpr int kSelCap = 2048;
constexpr int kSelBatch = 8;  // float4 of logits per thread per batch (row scan)
constexpr int kSelQuads = 256;  // quadrants read directly
constexpr int kSelQPer = 4;     // quadrant statistics per thread in registers

struct SelArgs {
  const float* logits;  // [M][V_high], bias added
  const float2* qstat;  // [M][nq]
  int nq, V_high, k;
  const int32_t* t2f;
  int32_t* out_ids;
  float* out_probs;
  float inv_tau;
};

__global__ void __launch_bounds__(kSelThreads, 1)
    rows_select_kernel(SelArgs a) {
  __shared__ float red[kSelWarps];
  __shared__ unsigned wkey[32];  // float_key of each group's maximum (0: empty)
  __shared__ entry_key surv[kSelCap];
  __shared__ float surv_s[kSelCap];
  __shared__ unsigned hist[256];
  __shared__ int cquad[kSelQuads];
  __shared__ int s_cnt, s_need, s_digit, s_nq;
  __shared__ unsigned s_lkey;
  grid_dependency_wait();
  grid_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = blockIdx.x, k = a.k;
  const float2* qs = a.qstat + (size_t)m * a.nq;
  const float* row = a.logits + (size_t)m * a.V_high;
  const bool vec = ((a.V_high & 3) == 0) &&
                   ((reinterpret_cast<uintptr_t>(a.logits) & 15) == 0);


  // the first kSelQPer * kSelThreads quadrants' statistics stay in
  // registers (one L2 round trip); any beyond are read again per pass
  float2 st[kSelQPer];
#pragma unroll
  for (int r = 0; r < kSelQPer; ++r) {
    const int q = tid + r * kSelThreads;
    st[r] = q < a.nq ? __ldcg(&qs[q]) : make_float2(-INFINITY, 0.f);
  }
  auto stat = [&](int q, int r) { return r < kSelQPer ? st[r] : __ldcg(&qs[q]); };
  if (tid < 32) wkey[tid] = 0u;
  if (tid == 0) { s_cnt = 0; s_nq = 0; }
  __syncthreads();
  float lm = -INFINITY;
  unsigned gk = 0u;  // this thread's largest quadrant maximum (0: none)
#pragma unroll 1
  for (int q = tid, r = 0; q < a.nq; q += kSelThreads, ++r) {
    const float mq = stat(q, r).x;
    lm = fmaxf(lm, mq);
    if (mq > -INFINITY) gk = max(gk, float_key(mq));
  }
  // thread t holds quadrants t + 1024 j, all = t mod 32 = its lane
  if (gk) atomicMax(&wkey[lane], gk);
  const float mg = block_max<kSelThreads>(lm, red);  // (its barriers publish wkey)
  float ls = 0.f;
#pragma unroll 1
  for (int q = tid, r = 0; q < a.nq; q += kSelThreads, ++r) {
    const float2 sq = stat(q, r);
    if (sq.y > 0.f) ls += sq.y * __expf(sq.x - mg);
  }
  if (warp == 0) {
    // L: the k-th largest group maximum (ties by group index); an empty
    // group (key 0) among the k best makes L = 0, which keeps every key
    const unsigned v = wkey[lane];
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const unsigned u = __shfl_sync(~0u, v, j);
      rank += (u > v) || (u == v && j < lane);
    }
    if (rank == k - 1) s_lkey = v;
  }
  const float sg = block_sum<kSelThreads>(ls, red);  // (its barriers publish s_lkey)
  const unsigned lkey = s_lkey;
  // the quadrants whose maximum reaches L
#pragma unroll 1
  for (int q = tid, r = 0; q < a.nq; q += kSelThreads, ++r) {
    const float mq = stat(q, r).x;
    if (mq > -INFINITY && float_key(mq) >= lkey) {
      const int p = atomicAdd(&s_nq, 1);
      if (p < kSelQuads) cquad[p] = q;
    }
  }
  __syncthreads();
  const int nquad = s_nq;

  auto score = [&](int i) { return __fmul_rn(__ldcg(row + i), a.inv_tau); };
  auto fid = [&](int i) { return a.t2f ? __ldg(a.t2f + i) : i; };
  auto keep_id = [&](int f, float sv) {
    const int p = atomicAdd(&s_cnt, 1);
    if (p < kSelCap) {
      surv[p] = make_key(sv, f);
      surv_s[p] = sv;
    }
  };
  auto keep = [&](int i, float sv) { keep_id(fid(i), sv); };
  if (nquad <= kSelQuads) {
    // logit and full id loaded together: one round trip
    for (int j = tid; j < nquad * 32; j += kSelThreads) {
      const int i = cquad[j >> 5] * 32 + (j & 31);
      if (i < a.V_high) {
        const float l = __ldcg(row + i);
        const int f = fid(i);
        const float sv = __fmul_rn(l, a.inv_tau);
        if (float_key(sv) >= lkey) keep_id(f, sv);
      }
    }
  } else if (vec) {
    float4 x[kSelBatch];
    for (int i0 = 4 * tid; i0 < a.V_high; i0 += 4 * kSelThreads * kSelBatch) {
#pragma unroll
      for (int b = 0; b < kSelBatch; ++b) {
        const int i = i0 + 4 * kSelThreads * b;
        x[b] = i < a.V_high ? __ldcg(reinterpret_cast<const float4*>(row + i))
                            : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int b = 0; b < kSelBatch; ++b) {
        const int i = i0 + 4 * kSelThreads * b;
        const float v[4] = {__fmul_rn(x[b].x, a.inv_tau), __fmul_rn(x[b].y, a.inv_tau),
                            __fmul_rn(x[b].z, a.inv_tau), __fmul_rn(x[b].w, a.inv_tau)};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i < a.V_high && float_key(v[e]) >= lkey) keep(i + e, v[e]);
      }
    }
  } else {
    for (int i = tid; i < a.V_high; i += kSelThreads) {
      const float sv = score(i);
      if (float_key(sv) >= lkey) keep(i, sv);
    }
  }
  __syncthreads();
  int S = s_cnt;

  if (S > kSelCap) {
    // radix select of the k-th best key among those reaching L, most
    // significant digit first
    entry_key prefix = 0ull, pmask = 0ull;
    int need = k;
    for (int p = 7; p >= 0; --p) {
      if (tid < 256) hist[tid] = 0u;
      __syncthreads();
      for (int i = tid; i < a.V_high; i += kSelThreads) {
        const float sv = score(i);
        if (float_key(sv) < lkey) continue;
        const entry_key key = make_key(sv, fid(i));
        if ((key & pmask) == prefix) atomicAdd(&hist[(unsigned)(key >> (8 * p)) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l holds digits 255-8l .. 248-8l; find the digit where the
        // count of larger-or-equal digits first reaches need
        unsigned c[8], tot = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) { c[e] = hist[255 - 8 * lane - e]; tot += c[e]; }
        unsigned before = tot;  // inclusive scan over lanes, then exclusive
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(~0u, before, o);
          if (lane >= o) before += y;
        }
        before -= tot;
        if (before < (unsigned)need && before + tot >= (unsigned)need) {
          unsigned run = before;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (run + c[e] >= (unsigned)need) {
              s_digit = 255 - 8 * lane - e;
              s_need = need - (int)run;
              break;
            }
            run += c[e];
          }
        }
      }
      __syncthreads();
      prefix |= (entry_key)(unsigned)s_digit << (8 * p);
      pmask |= 0xffull << (8 * p);
      need = s_need;
      __syncthreads();
    }
    // prefix is the k-th best key: collect the k keys at or above it
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    for (int i = tid; i < a.V_high; i += kSelThreads) {
      const float sv = score(i);
      if (float_key(sv) < lkey) continue;
      if (make_key(sv, fid(i)) >= prefix) keep(i, sv);
    }
    __syncthreads();
    S = min(s_cnt, k);
  }

  int32_t* ids = a.out_ids + (size_t)m * k;
  float* probs = a.out_probs + (size_t)m * k;
  for (int c = tid; c < S; c += kSelThreads) {
    const entry_key xk = surv[c];
    int rank = 0;
    for (int q = 0; q < S; ++q) rank += surv[q] > xk;
    if (rank < k) {
      ids[rank] = key_id(xk);
      probs[rank] = expf(surv_s[c] - mg) / sg;
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

// Workspace of the tensor-core path: the shared header (error word at byte
// 128, per-row tickets from byte 1024), then per-row partials of the top-k
// kernel, then the fp32 logits.
struct TcLayout {
  size_t tickets, part, qstat, logits, total;
};
static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
static int row_parts(int V_high) { return (V_high + kRowSpan - 1) / kRowSpan; }
static int quadrants(int V_high) { return 4 * ((V_high + kTcTileRows - 1) / kTcTileRows); }
static TcLayout tc_layout(int M, int V_high, int k) {
  TcLayout L;
  L.tickets = kHeadRowTicketOffset;
  L.part = kHeadTicketBytes;
  L.qstat = L.part + round256((size_t)M * row_parts(V_high) * (2 + 3 * k) * 4);
  L.logits = L.qstat + round256((size_t)M * quadrants(V_high) * sizeof(float2));
  L.total = L.logits + (size_t)M * V_high * 4;
  return L;
}

size_t head_tc_workspace(int M, int V_high, int k) {
  return tc_layout(M, V_high, k).total;
}

vt_status head_tc(const uint16_t* H, int M, int d, int64_t ldh,
                  const uint16_t* W, int V_high, const int32_t* t2f, int k,
                  const HeadOpts& opt, int32_t* out_ids, float* out_probs,
                  float* out_logits, void* ws, const DeviceInfo& di,
                  cudaStream_t s) {
  if (M > 256) return fail(VT_ERR_UNSUPPORTED, "head_tc: M > 256");
  const TcLayout L = tc_layout(M, V_high, k);
  char* wsb = static_cast<char*>(ws);
  unsigned* err = reinterpret_cast<unsigned*>(wsb + 128);
  float* logits = out_logits ? out_logits : reinterpret_cast<float*>(wsb + L.logits);
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
  a.bias = opt.bias;
  a.err = err;
  // top-k calls: quadrant statistics for rows_select_kernel; sampling calls
  // score every logit with its noise in rows_topk_kernel instead
  const bool stats = !opt.sample;
  a.qstat = stats ? reinterpret_cast<float2*>(wsb + L.qstat) : nullptr;
  a.nq = quadrants(V_high);
  a.inv_tau = 1.0f / opt.tau;
  // Few tiles (two per SM or fewer): split each tile's K stages between the
  // two CTAs of a cluster, so twice as many SMs stream W_high; the exchange
  // buffer of the partner's partial sums takes N * 64 * 4 bytes.
  const int ntiles = (V_high + kTcTileRows - 1) / kTcTileRows;
  const int natoms = (d + kTcBlockK - 1) / kTcBlockK;
  a.ksplit = 2 * ntiles <= di.num_sms && natoms >= 2 * kTcMaxAtoms ? 1 : 0;
  const int xbytes = a.ksplit ? a.N * 64 * 4 : 0;
  // K atoms per stage: the widest (up to kTcMaxAtoms) that still leaves
  // kTcMinStages stages in shared memory.
  const int atom_bytes = kTcABytes + a.N * kTcBlockK * 2;
  const int fit = (di.max_smem_optin - 4096 - xbytes) / atom_bytes;  // atoms that fit
  a.atoms = std::max(1, std::min(kTcMaxAtoms, fit / kTcMinStages));
  const int stage_bytes = a.atoms * atom_bytes;
  a.stages = std::min<int>(kTcMaxStages, fit / a.atoms);
  if (a.stages < 2) return fail(VT_ERR_UNSUPPORTED, "head_tc: stages do not fit");
  CUtensorMap tmW, tmH;
  if (!make_map(&tmW, W, (uint64_t)V_high, (uint64_t)d, (uint64_t)d, kTcTileRows) ||
      !make_map(&tmH, H, (uint64_t)M, (uint64_t)d, (uint64_t)ldh, (uint32_t)a.N))
    return fail(VT_ERR_CUDA, "head_tc: cuTensorMapEncodeTiled failed");
  if (!allow_max_smem(head_tc_gemm_kernel, di)) return VT_ERR_CUDA;
  // Whole tiles: as many waves of tiles as the SMs need, spread evenly
  // (256 tiles on 152 SMs: 128 CTAs of two tiles rather than 104 of two and
  // 48 of one, so no SM streams alone at the end; 512 tiles: 128 of four).
  const int waves = (ntiles + di.num_sms - 1) / di.num_sms;
  const int grid = a.ksplit ? 2 * ntiles : (ntiles + waves - 1) / waves;
  const int smem = a.stages * stage_bytes + xbytes + 1024;
  // a programmatic dependent of the work ahead of it in the stream; with the
  // K split, in clusters of two CTAs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.ksplit ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, head_tc_gemm_kernel, tmW, tmH, a);
  if (e != cudaSuccess)
    return fail(VT_ERR_CUDA, std::string("head_tc_gemm_kernel: ") + cudaGetErrorString(e));
  vt_status st = launch_status("head_tc_gemm_kernel");
  if (st != VT_OK) return st;
  if (stats) {
    SelArgs sa;
    sa.logits = logits;
    sa.qstat = a.qstat;
    sa.nq = a.nq;
    sa.V_high = V_high;
    sa.k = k;
    sa.t2f = t2f;
    sa.out_ids = out_ids;
    sa.out_probs = out_probs;
    sa.inv_tau = a.inv_tau;
    // a programmatic dependent of the GEMM, like the per-row kernel below
    const cudaError_t e3 = launch_dependent(rows_select_kernel, dim3(M),
                                            dim3(kSelThreads), 0, s, sa);
    if (e3 != cudaSuccess)
      return fail(VT_ERR_CUDA, std::string("rows_select_kernel: ") + cudaGetErrorString(e3));
    return launch_status("rows_select_kernel");
  }
  const int P = row_parts(V_high);
  if (P * k > kRowSurvivors)
    return fail(VT_ERR_UNSUPPORTED, "head_tc: V_high * k too large for the row merge");
  RowArgs r;
  r.logits = logits;
  r.V_high = V_high;
  r.k = k;
  r.P = P;
  r.t2f = t2f;
  r.out_ids = out_ids;
  r.out_probs = out_probs;
  r.tickets = reinterpret_cast<unsigned*>(wsb + L.tickets);
  r.part = reinterpret_cast<float*>(wsb + L.part);
  r.inv_tau = 1.0f / opt.tau;
  r.sample = opt.sample;
  r.seed = opt.seed;
  r.offset = opt.offset;
  r.row_ids = opt.row_ids;
  // a programmatic dependent of the GEMM: launched (and possibly resident)
  // early; each CTA waits for the GEMM's logits in griddepcontrol.wait
  if (!allow_max_smem(rows_topk_kernel, di)) return VT_ERR_CUDA;
  const cudaError_t e2 = launch_dependent(rows_topk_kernel, dim3(P, M),
                                          dim3(kRowThreads), kRowSmem, s, r);
  if (e2 != cudaSuccess)
    return fail(VT_ERR_CUDA, std::string("rows_topk_kernel: ") + cudaGetErrorString(e2));
  return launch_status("rows_topk_kernel");
}

}  // namespace vt
