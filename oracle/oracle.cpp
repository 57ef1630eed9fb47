// Plain CPU oracle for the frequency-ranked trimmed drafter head.
//
// TEST INFRASTRUCTURE ONLY.  Nothing under frequency_ranked_drafter_gb300/
// links, loads or calls this file; only tests/, __graft_entry__.smoke() and
// the cpu_baseline / reference leg of bench.py may do so.  It shares no code,
// header, table or helper with the CUDA library.
//
// Every function is the plain definition of one step, written for a reader
// who checks it against the pages by eye: single-threaded, no blocking, no
// fusion, exact integer arithmetic and fp64 for everything that is floating
// point.  Sources (page title, then section):
//   [VT]  "VocabTrim: Memory-Efficient Vocabulary Pruning for Speculative
//         Decoding" (skill page, English and Japanese copies), Implementation
//         Steps 1-4.
//   [FR]  "FR-Spec: Accelerating Large-Vocabulary Language Models via
//         Frequency-Ranked Speculative Sampling" (ACL 2025 paper notes),
//         Method > Key design "frequency-ranked vocabulary compression".
//
// Readings where the pages are silent (each one also listed in the design
// notes of the repository):
//   * selection ties: count descending, then lower token id first (the pages
//     sort a dict by count only, which leaves ties in first-seen order);
//   * ids never seen are candidates with count 0, so the kept list always has
//     exactly V_high entries;
//   * ids outside [0, V) are not counted; they are reported separately and do
//     not enter the coverage denominator;
//   * top-k ties: larger logit first, then lower full-vocabulary id;
//   * drawing from the trimmed distribution ([VT] Step 4 samples with
//     multinomial) is done by the Gumbel-max rule, which draws from the same
//     distribution: the noise of each token comes from the counter-based
//     generator Philox4x32-10 keyed by (seed, step offset, hidden state,
//     full-vocabulary id), so a token's noise does not depend on which other
//     tokens were kept.  The k best of logit/T + noise are k draws without
//     replacement (k = 1: one draw).
//
// Build: g++ -O2 -std=c++17 -shared -fPIC oracle.cpp -o liboracle.so
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <vector>

namespace {

// bf16 is the upper half of an IEEE binary32; widening to double is exact.
double bf16_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Philox4x32-10: the counter-based generator of Salmon, Moraes, Dror and
// Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011).  Ten rounds;
// a round multiplies counter words 0 and 2 by the two round multipliers
// (64-bit products split into high and low halves) and mixes in the key;
// the key advances by the two Weyl increments between rounds.
void philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                   uint32_t out[4]) {
  const uint64_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  const uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
  uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  uint32_t k[2] = {key_in[0], key_in[1]};
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k[0] += kWeyl0;
      k[1] += kWeyl1;
    }
    const uint64_t p0 = kMul0 * c[0];
    const uint64_t p1 = kMul1 * c[2];
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32);
    const uint32_t lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32);
    const uint32_t lo1 = static_cast<uint32_t>(p1);
    const uint32_t n0 = hi1 ^ c[1] ^ k[0];
    const uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
  for (int i = 0; i < 4; ++i) out[i] = c[i];
}

// Gumbel noise of token `full_id` for hidden state m at step (seed, offset):
// x = word 0 of Philox4x32-10 with counter (full_id, m, offset low, offset
// high) and key (seed low, seed high); u = ((x >> 9) + 1/2) / 2^23, which
// lies in (0, 1) and is exact in binary32; g = -log(-log(u)).
double gumbel_noise(uint64_t seed, uint64_t offset, int32_t m, int32_t full_id) {
  const uint32_t ctr[4] = {static_cast<uint32_t>(full_id), static_cast<uint32_t>(m),
                           static_cast<uint32_t>(offset),
                           static_cast<uint32_t>(offset >> 32)};
  const uint32_t key[2] = {static_cast<uint32_t>(seed),
                           static_cast<uint32_t>(seed >> 32)};
  uint32_t x[4];
  philox4x32_10(ctr, key, x);
  const double u = (static_cast<double>(x[0] >> 9) + 0.5) / 8388608.0;
  return -std::log(-std::log(u));
}

}  // namespace

extern "C" {

// Histogram of a token stream.  [VT] Step 1 counts each id into a dict,
// token_counts[id] = token_counts.get(id, 0) + 1; [FR] counts corpus tokens.
// counts[V] is OVERWRITTEN with the dict densified over 0..V-1.
// *n_invalid receives the number of ids outside [0, V).
int oracle_count_tokens(const int32_t* tokens, int64_t n, int32_t V,
                        uint64_t* counts, uint64_t* n_invalid) {
  if (V <= 0 || n < 0 || counts == nullptr) return 1;
  std::unordered_map<int32_t, uint64_t> token_counts;
  uint64_t invalid = 0;
  for (int64_t i = 0; i < n; ++i) {
    int32_t id = tokens[i];
    if (id < 0 || id >= V) {
      ++invalid;
      continue;
    }
    token_counts[id] += 1;
  }
  for (int32_t id = 0; id < V; ++id) counts[id] = 0;
  for (const auto& kv : token_counts) counts[kv.first] = kv.second;
  if (n_invalid) *n_invalid = invalid;
  return 0;
}

// Vocabulary selection and the two index maps.  [VT] Step 2: sort by count
// descending, keep the first target_vocab_size entries; the trimmed index of
// an id is its position in that sorted list (full_to_trimmed /
// trimmed_to_full); coverage = selected_count / total_count.
// Outputs: t2f[V_high], f2t[V] (-1 for dropped ids), *kept, *total, and
// *coverage = kept / total as one IEEE double division (NaN when total = 0).
int oracle_select_vocab(const uint64_t* counts, int32_t V, int32_t V_high,
                        int32_t* t2f, int32_t* f2t, uint64_t* kept,
                        uint64_t* total, double* coverage) {
  if (V <= 0 || V_high <= 0 || V_high > V) return 1;
  struct Entry {
    uint64_t count;
    int32_t id;
  };
  std::vector<Entry> items;
  items.reserve(V);
  for (int32_t id = 0; id < V; ++id) items.push_back({counts[id], id});
  std::sort(items.begin(), items.end(), [](const Entry& a, const Entry& b) {
    if (a.count != b.count) return a.count > b.count;  // more frequent first
    return a.id < b.id;                                // tie: lower id first
  });
  for (int32_t id = 0; id < V; ++id) f2t[id] = -1;
  uint64_t selected_count = 0;
  for (int32_t i = 0; i < V_high; ++i) {
    t2f[i] = items[i].id;
    f2t[items[i].id] = i;
    selected_count += items[i].count;
  }
  uint64_t total_count = 0;
  for (int32_t id = 0; id < V; ++id) total_count += counts[id];
  if (kept) *kept = selected_count;
  if (total) *total = total_count;
  if (coverage)
    *coverage = static_cast<double>(selected_count) /
                static_cast<double>(total_count);
  return 0;
}

// LM-head reconstruction.  [VT] Step 3: trimmed_weight =
// original_weight[selected_indices, :], weight stored [vocab, hidden].
// A row whose index is outside [0, V) is written as zeros (return value 2).
int oracle_gather_rows(const uint16_t* W, int64_t V, int32_t d,
                       const int32_t* t2f, int32_t V_high, uint16_t* W_high) {
  int rc = 0;
  for (int32_t i = 0; i < V_high; ++i) {
    int64_t src = t2f[i];
    uint16_t* dst = W_high + static_cast<int64_t>(i) * d;
    if (src < 0 || src >= V) {
      std::memset(dst, 0, sizeof(uint16_t) * d);
      rc = 2;
      continue;
    }
    std::memcpy(dst, W + src * d, sizeof(uint16_t) * d);
  }
  return rc;
}

// Bias of the kept rows.  [VT] Step 3 copies the old head's bias with the
// kept ids (new_bias[i] = old_bias[trimmed_to_full[i]]) when the head has
// one.  b_high[i] = b[t2f[i]]; ids outside [0, V) give 0.  Returns the
// number of such ids.
int64_t oracle_gather_bias(const float* b, int64_t V, const int32_t* t2f,
                           int32_t V_high, float* b_high) {
  int64_t bad = 0;
  for (int32_t i = 0; i < V_high; ++i) {
    const int64_t src = t2f[i];
    if (src < 0 || src >= V) {
      b_high[i] = 0.0f;
      ++bad;
      continue;
    }
    b_high[i] = b[src];
  }
  return bad;
}

// Trimmed projection.  [FR] Key design: the draft LM head projects onto the
// V_high kept rows only (weight d x 128k -> d x 32k); [VT] Step 4 runs the
// reconstructed Linear.  logits[m][i] = sum_j H[m][j] * W_high[i][j], every
// product exact in double, summed in j order.  H rows are ldh elements apart.
int oracle_head_logits(const uint16_t* H, int32_t M, int32_t d, int64_t ldh,
                       const uint16_t* W_high, int32_t V_high,
                       double* logits) {
  for (int32_t m = 0; m < M; ++m) {
    const uint16_t* h = H + static_cast<int64_t>(m) * ldh;
    for (int32_t i = 0; i < V_high; ++i) {
      const uint16_t* w = W_high + static_cast<int64_t>(i) * d;
      double acc = 0.0;
      for (int32_t j = 0; j < d; ++j)
        acc += bf16_to_double(h[j]) * bf16_to_double(w[j]);
      logits[static_cast<int64_t>(m) * V_high + i] = acc;
    }
  }
  return 0;
}

// One draft step of the trimmed head for M hidden states.
//   logits   : as oracle_head_logits;
//   softmax  : over the V_high trimmed logits only ([VT] Step 4
//              trimmed_probs = softmax(drafter_logits); [FR] "softmax is
//              computed on the subset only"), p_i = exp(l_i - max) / sum_j
//              exp(l_j - max) in double;
//   top-k    : the k largest logits (ties: lower full id first), in
//              descending order; k = 1 is the greedy argmax;
//   remap    : trimmed index -> full id through t2f ([VT] Step 4 "REMAP");
//              t2f == nullptr means the identity (the untrimmed head).
// Outputs per row m (each nullable): ids[m*k+r], probs[m*k+r],
// top_logits[m*k+r], trimmed_idx[m*k+r], row_max[m], row_sumexp[m].
int oracle_draft_head(const uint16_t* H, int32_t M, int32_t d, int64_t ldh,
                      const uint16_t* W_high, int32_t V_high,
                      const int32_t* t2f, int32_t k, int32_t* ids,
                      double* probs, double* top_logits, int32_t* trimmed_idx,
                      double* row_max, double* row_sumexp) {
  if (M < 0 || d <= 0 || V_high <= 0 || k <= 0 || k > V_high) return 1;
  std::vector<double> logits(static_cast<size_t>(V_high));
  std::vector<int32_t> order(static_cast<size_t>(V_high));
  for (int32_t m = 0; m < M; ++m) {
    oracle_head_logits(H + static_cast<int64_t>(m) * ldh, 1, d, ldh, W_high,
                       V_high, logits.data());
    double mx = logits[0];
    for (int32_t i = 1; i < V_high; ++i) mx = std::max(mx, logits[i]);
    double sumexp = 0.0;
    for (int32_t i = 0; i < V_high; ++i) sumexp += std::exp(logits[i] - mx);

    auto full_id = [&](int32_t i) { return t2f ? t2f[i] : i; };
    for (int32_t i = 0; i < V_high; ++i) order[i] = i;
    std::partial_sort(order.begin(), order.begin() + k, order.end(),
                      [&](int32_t a, int32_t b) {
                        if (logits[a] != logits[b]) return logits[a] > logits[b];
                        return full_id(a) < full_id(b);
                      });
    for (int32_t r = 0; r < k; ++r) {
      const int32_t i = order[r];
      const int64_t o = static_cast<int64_t>(m) * k + r;
      if (ids) ids[o] = full_id(i);
      if (probs) probs[o] = std::exp(logits[i] - mx) / sumexp;
      if (top_logits) top_logits[o] = logits[i];
      if (trimmed_idx) trimmed_idx[o] = i;
    }
    if (row_max) row_max[m] = mx;
    if (row_sumexp) row_sumexp[m] = sumexp;
  }
  return 0;
}

// Philox4x32-10 output block for one (counter, key), for the pins.
int oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key,
                         uint32_t* out) {
  philox4x32_10(ctr, key, out);
  return 0;
}

// Gumbel noise for n full ids (see gumbel_noise), for the pins.
int oracle_gumbel_noise(uint64_t seed, uint64_t offset, int32_t m,
                        const int32_t* full_ids, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = gumbel_noise(seed, offset, m, full_ids[i]);
  return 0;
}

// One draft step with the head's options.
//   logits   : l_i = sum_j H[m][j] * W_high[i][j] + b_i, where b = bias_high
//              (the kept rows' bias, [VT] Step 3's optional bias copy;
//              nullptr = no bias), every product exact in double;
//   temper   : s_i = l_i / temperature (temperature > 0; 1 = plain logits);
//   softmax  : p_i = exp(s_i - max s) / sum_j exp(s_j - max s), over the kept
//              rows only, in double;
//   select   : mode 0 (top-k): the k largest s_i; mode 1 (sample): the k
//              largest s_i + g_i with g_i = gumbel_noise(seed, offset, m,
//              full id of i) (m counted from m_base, the row of the first
//              hidden state in the caller's batch): one draw from p for k = 1 (Gumbel-max), k
//              draws without replacement for k > 1; ties in either key go
//              to the lower full id; descending;
//   remap    : trimmed index -> full id through t2f (nullptr = identity).
// Outputs per row m (each nullable): ids[m*k+r], probs[m*k+r] = p of the
// chosen entry, scores[m*k+r] = its selection key, top_logits[m*k+r] = its
// l, trimmed_idx[m*k+r], row_max[m] = max s, row_sumexp[m].
int oracle_draft_head_ex(const uint16_t* H, int32_t M, int32_t d, int64_t ldh,
                         const uint16_t* W_high, int32_t V_high,
                         const int32_t* t2f, const float* bias_high,
                         double temperature, int32_t mode, uint64_t seed,
                         uint64_t offset, int32_t m_base, int32_t k, int32_t* ids,
                         double* probs, double* scores, double* top_logits,
                         int32_t* trimmed_idx, double* row_max,
                         double* row_sumexp) {
  if (M < 0 || d <= 0 || V_high <= 0 || k <= 0 || k > V_high) return 1;
  if (!(temperature > 0.0) || (mode != 0 && mode != 1)) return 1;
  std::vector<double> logits(static_cast<size_t>(V_high));
  std::vector<double> s(static_cast<size_t>(V_high));
  std::vector<double> key(static_cast<size_t>(V_high));
  std::vector<int32_t> order(static_cast<size_t>(V_high));
  auto full_id = [&](int32_t i) { return t2f ? t2f[i] : i; };
  for (int32_t m = 0; m < M; ++m) {
    oracle_head_logits(H + static_cast<int64_t>(m) * ldh, 1, d, ldh, W_high,
                       V_high, logits.data());
    for (int32_t i = 0; i < V_high; ++i) {
      logits[i] += bias_high ? static_cast<double>(bias_high[i]) : 0.0;
      s[i] = logits[i] / temperature;
    }
    double mx = s[0];
    for (int32_t i = 1; i < V_high; ++i) mx = std::max(mx, s[i]);
    double sumexp = 0.0;
    for (int32_t i = 0; i < V_high; ++i) sumexp += std::exp(s[i] - mx);
    for (int32_t i = 0; i < V_high; ++i)
      key[i] = s[i] + (mode == 1 ? gumbel_noise(seed, offset, m_base + m, full_id(i)) : 0.0);

    for (int32_t i = 0; i < V_high; ++i) order[i] = i;
    std::partial_sort(order.begin(), order.begin() + k, order.end(),
                      [&](int32_t a, int32_t b) {
                        if (key[a] != key[b]) return key[a] > key[b];
                        return full_id(a) < full_id(b);
                      });
    for (int32_t r = 0; r < k; ++r) {
      const int32_t i = order[r];
      const int64_t o = static_cast<int64_t>(m) * k + r;
      if (ids) ids[o] = full_id(i);
      if (probs) probs[o] = std::exp(s[i] - mx) / sumexp;
      if (scores) scores[o] = key[i];
      if (top_logits) top_logits[o] = logits[i];
      if (trimmed_idx) trimmed_idx[o] = i;
    }
    if (row_max) row_max[m] = mx;
    if (row_sumexp) row_sumexp[m] = sumexp;
  }
  return 0;
}

// Full-vocabulary draft distribution of one draft step.  [FR] Method > Key
// design: only the draft step changes; verification still uses the full
// target model and accepts or rejects draft tokens so that the output
// follows the target's distribution exactly (rejection sampling), which
// compares the target's and the draft's probabilities over the whole
// vocabulary.  The trimmed draft gives dropped ids probability 0:
//   q[m][f] = p[m][i] if f = t2f[i] (a kept id), 0 otherwise,
// with p the softmax((logit + bias) / T) over the kept rows (as in
// oracle_draft_head_ex).  q is [M][V]; t2f == nullptr is the identity
// (V == V_high).
int oracle_draft_q(const uint16_t* H, int32_t M, int32_t d, int64_t ldh,
                   const uint16_t* W_high, int32_t V_high, const int32_t* t2f,
                   const float* bias_high, double temperature, int32_t V,
                   double* q) {
  if (M < 0 || d <= 0 || V_high <= 0 || V < V_high || !(temperature > 0.0))
    return 1;
  if (!t2f && V != V_high) return 1;
  std::vector<double> s(static_cast<size_t>(V_high));
  for (int32_t m = 0; m < M; ++m) {
    oracle_head_logits(H + static_cast<int64_t>(m) * ldh, 1, d, ldh, W_high,
                       V_high, s.data());
    for (int32_t i = 0; i < V_high; ++i)
      s[i] = (s[i] + (bias_high ? static_cast<double>(bias_high[i]) : 0.0)) /
             temperature;
    double mx = s[0];
    for (int32_t i = 1; i < V_high; ++i) mx = std::max(mx, s[i]);
    double sumexp = 0.0;
    for (int32_t i = 0; i < V_high; ++i) sumexp += std::exp(s[i] - mx);
    double* qm = q + static_cast<int64_t>(m) * V;
    for (int32_t f = 0; f < V; ++f) qm[f] = 0.0;
    for (int32_t i = 0; i < V_high; ++i) {
      const int32_t f = t2f ? t2f[i] : i;
      if (f < 0 || f >= V) return 2;
      qm[f] = std::exp(s[i] - mx) / sumexp;
    }
  }
  return 0;
}

}  // extern "C"
