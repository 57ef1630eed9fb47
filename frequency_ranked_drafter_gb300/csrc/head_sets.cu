// vt_draft_head_sets — one draft step for hidden states that use different
// kept vocabularies.
//
// "FR-Spec: Accelerating Large-Vocabulary Language Models via
// Frequency-Ranked Speculative Sampling", Limitations: the kept vocabulary is
// a single static set counted over a whole corpus, and vocabularies chosen
// per domain or per request are left as future work.  Here each set (its own
// t2f and W_high, built by the same offline steps from its own token stream)
// serves the hidden states assigned to it: hidden state m is scored against
// set s_m exactly as vt_draft_head_ex scores it alone, and when drawing its
// noise index is still its row m in this call.
//
// Rows are grouped by set on the host.  One small kernel gathers every
// row's hidden state into contiguous memory, set by set (and writes the row
// numbers for the noise); then, for each set used, the head runs on that
// set's rows (GEMV for one row, the tensor-core path for more), each head a
// programmatic dependent of the one before (its weights start streaming
// while the previous set's selection finishes); a last small kernel
// scatters all ids and probabilities back to their rows.  (With a gather and
// a scatter around each set's head, two sets of 32768 rows at M = 4 took
// 107.6 us.)
#include <vector>

#include "head_common.cuh"

namespace vt {
namespace {

constexpr int kSetsMaxRows = 256;

struct RowList {
  int32_t n;
  int32_t rows[kSetsMaxRows];
};

__global__ void sets_gather_kernel(const uint16_t* __restrict__ H, int64_t ldh,
                                   int d, RowList L, uint16_t* __restrict__ Hg,
                                   int32_t* __restrict__ row_ids) {
  const int j = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(H + (int64_t)L.rows[j] * ldh);
  uint4* dst = reinterpret_cast<uint4*>(Hg + (int64_t)j * d);
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) dst[c] = src[c];
  if (threadIdx.x == 0) row_ids[j] = L.rows[j];
}

__global__ void sets_scatter_kernel(const int32_t* __restrict__ ids_g,
                                    const float* __restrict__ probs_g,
                                    RowList L, int k,
                                    int32_t* __restrict__ out_ids,
                                    float* __restrict__ out_probs) {
  for (int t = threadIdx.x; t < L.n * k; t += blockDim.x) {
    const int j = t / k, r = t - j * k;
    if (!VT_CHECKED(L.rows[j] >= 0 && L.rows[j] < kSetsMaxRows)) continue;
    out_ids[(int64_t)L.rows[j] * k + r] = ids_g[t];
    out_probs[(int64_t)L.rows[j] * k + r] = probs_g[t];
  }
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct SetsLayout {
  size_t head, Hg, ids, probs, rows, total;
};

SetsLayout sets_layout(int32_t M, int32_t d, int32_t k, int32_t S,
                       const int32_t* V_high_sets) {
  size_t head = 0;
  for (int s = 0; s < S; ++s) {
    head = std::max(head, vt_draft_head_workspace_size(M, V_high_sets[s], k));
    head = std::max(head, vt_draft_head_workspace_size(1, V_high_sets[s], k));
  }
  SetsLayout L;
  L.head = 0;
  L.Hg = round256(head);
  L.ids = L.Hg + round256((size_t)M * d * 2);
  L.probs = L.ids + round256((size_t)M * k * 4);
  L.rows = L.probs + round256((size_t)M * k * 4);
  L.total = L.rows + round256((size_t)M * 4);
  return L;
}

}  // namespace
}  // namespace vt

extern "C" size_t vt_draft_head_sets_workspace_size(int32_t M, int32_t d,
                                                    int32_t k, int32_t S,
                                                    const int32_t* V_high_sets) {
  if (M <= 0 || d <= 0 || k <= 0 || S <= 0 || !V_high_sets) return 0;
  for (int s = 0; s < S; ++s)
    if (V_high_sets[s] <= 0) return 0;
  return vt::sets_layout(M, d, k, S, V_high_sets).total;
}

extern "C" vt_status vt_draft_head_sets(
    const uint16_t* H, int32_t M, int32_t d, int64_t ldh,
    const int32_t* set_of_row, int32_t S, const uint16_t* const* W_high_sets,
    const int32_t* V_high_sets, const int32_t* const* t2f_sets,
    const float* const* bias_sets, int32_t k, const vt_head_options* opts,
    int32_t* out_ids, float* out_probs, void* ws, size_t ws_bytes,
    void* stream) {
  using namespace vt;
  if (!H || !set_of_row || !W_high_sets || !V_high_sets || !out_ids || !out_probs)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head_sets: null pointer");
  if (M < 1 || M > kSetsMaxRows || S < 1)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head_sets: need 1 <= M <= 256, S >= 1");
  if (d < 8 || d > 16384 || d % 8 != 0 || ldh < d || ldh % 8 != 0 || !aligned(H, 16))
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_head_sets: need d % 8 == 0, ldh >= d, ldh % 8 == 0, H 16B aligned");
  if (k < 1 || k > kTopKMax)
    return fail(VT_ERR_INVALID_ARG, "vt_draft_head_sets: need 1 <= k <= 32");
  // every set is checked before anything is launched
  for (int s = 0; s < S; ++s) {
    if (!W_high_sets[s] || !aligned(W_high_sets[s], 16) || V_high_sets[s] < k)
      return fail(VT_ERR_INVALID_ARG,
                  "vt_draft_head_sets: every set needs a 16B-aligned W_high and V_high >= k");
    if (bias_sets && bias_sets[s] && !aligned(bias_sets[s], 4))
      return fail(VT_ERR_INVALID_ARG, "vt_draft_head_sets: bias not 4B aligned");
  }
  if (opts && opts->bias_high)
    return fail(VT_ERR_INVALID_ARG,
                "vt_draft_head_sets: biases go in bias_sets, one per set");
  std::vector<std::vector<int32_t>> rows(S);
  for (int m = 0; m < M; ++m) {
    if (set_of_row[m] < 0 || set_of_row[m] >= S)
      return fail(VT_ERR_INVALID_ARG, "vt_draft_head_sets: set index out of range");
    rows[set_of_row[m]].push_back(m);
  }
  const SetsLayout L = sets_layout(M, d, k, S, V_high_sets);
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total)
    return fail(VT_ERR_WORKSPACE,
                "vt_draft_head_sets: workspace missing, misaligned or too small");
  char* w = static_cast<char*>(ws);
  uint16_t* Hg = reinterpret_cast<uint16_t*>(w + L.Hg);
  int32_t* ids_g = reinterpret_cast<int32_t*>(w + L.ids);
  float* probs_g = reinterpret_cast<float*>(w + L.probs);
  int32_t* row_ids = reinterpret_cast<int32_t*>(w + L.rows);
  cudaStream_t st = (cudaStream_t)stream;
  // all rows, set by set: set s's rows sit at [first[s], first[s] + n_s)
  RowList rl;
  rl.n = M;
  std::vector<int> first(S, 0);
  for (int s = 0, j = 0; s < S; ++s) {
    first[s] = j;
    for (int32_t m : rows[s]) rl.rows[j++] = m;
  }
  sets_gather_kernel<<<M, 128, 0, st>>>(H, ldh, d, rl, Hg, row_ids);
  vt_status r = launch_status("sets_gather_kernel");
  if (r != VT_OK) return r;
  for (int s = 0; s < S; ++s) {
    const int n = (int)rows[s].size();
    if (n == 0) continue;
    const int j0 = first[s];
    vt_head_options o;
    if (opts) {
      o = *opts;
    } else {
      o.bias_high = nullptr;
      o.temperature = 1.0f;
      o.mode = VT_HEAD_TOPK;
      o.seed = 0;
      o.offset = 0;
    }
    o.bias_high = bias_sets ? bias_sets[s] : nullptr;
    r = draft_head_rows(Hg + (size_t)j0 * d, n, d, d, W_high_sets[s], V_high_sets[s],
                        t2f_sets ? t2f_sets[s] : nullptr, k, &o, row_ids + j0,
                        ids_g + (size_t)j0 * k, probs_g + (size_t)j0 * k, w + L.head,
                        L.Hg, stream);
    if (r != VT_OK) return r;
  }
  sets_scatter_kernel<<<1, 256, 0, st>>>(ids_g, probs_g, rl, k, out_ids, out_probs);
  return launch_status("sets_scatter_kernel");
}
