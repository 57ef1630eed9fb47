/*
 * vt.h — C ABI of the frequency-ranked trimmed drafter head (GB300, sm_103a).
 *
 * The library implements the data-parallel hot path of vocabulary trimming
 * for speculative-decoding drafters:
 *   offline build : token histogram -> top-V_high selection -> the two index
 *                   maps -> row gather of the kept lm_head rows;
 *   runtime head  : logits over the V_high kept rows only, fused with the
 *                   softmax over that subset, top-k, and the remap of the
 *                   chosen trimmed indices back to full-vocabulary ids.
 *
 * Sources (page title, then section):
 *   [VT] "VocabTrim: Memory-Efficient Vocabulary Pruning for Speculative
 *        Decoding" (skill page, English and Japanese copies), Architecture
 *        Overview and Implementation Steps 1-4.
 *   [FR] "FR-Spec: Accelerating Large-Vocabulary Language Models via
 *        Frequency-Ranked Speculative Sampling" (ACL 2025 paper notes),
 *        Method > Key design "frequency-ranked vocabulary compression".
 *
 * Conventions for every call
 *   - Pointers marked (device) must be device memory of the current CUDA
 *     device (or managed memory); (host) pointers are host memory.
 *   - bf16 tensors are passed as `const uint16_t*` holding the bf16 bit
 *     patterns; all matrices are row-major and densely packed.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call is asynchronous and stream-ordered; none synchronises, allocates
 *     or frees.  The caller owns every buffer.
 *   - Argument errors are detected on the host before anything is launched
 *     and are returned synchronously (VT_ERR_INVALID_ARG, VT_ERR_WORKSPACE,
 *     VT_ERR_UNSUPPORTED); nothing is written in that case.  A failed launch
 *     returns VT_ERR_CUDA.  vt_last_error() gives a one-line reason for the
 *     latest non-OK status returned on the calling thread.
 *   - Data errors inside buffers (ids outside the vocabulary) never trap:
 *     they are counted into an optional device counter and skipped.
 *   - Calls that take a workspace (`ws`) need one of at least the size the
 *     matching *_workspace_size function returns, 256-byte aligned.  Calls
 *     running concurrently (other streams) need distinct workspaces.
 *   - Error words.  Kernels that wait on other CTAs or on their own copies
 *     (vt_select_vocab's look-back, the head's merges and tensor-core
 *     pipeline) bound every wait (about a second).  A wait that gives up
 *     writes VT_ERR_TIMEOUT to the 32-bit word at byte 128 of the call's
 *     workspace and the kernel returns; the call's outputs are then
 *     incomplete.  The call itself has returned VT_OK by then (it is
 *     asynchronous): read the word after synchronising the stream.
 *     vt_host_step_run reads it for you and returns VT_ERR_TIMEOUT.  After a
 *     timeout the head's counters may be left set: zero-fill its workspace
 *     again before the next call.
 */
#ifndef VT_H_
#define VT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vt_status {
  VT_OK = 0,
  VT_ERR_INVALID_ARG = 1, /* null pointer, bad size or alignment */
  VT_ERR_CUDA = 2,        /* a CUDA runtime call or launch failed */
  VT_ERR_UNSUPPORTED = 3, /* valid but outside what this build supports */
  VT_ERR_WORKSPACE = 4,   /* workspace missing, too small or misaligned */
  VT_ERR_TIMEOUT = 5      /* a bounded device wait gave up (see error words) */
} vt_status;

/* Static string naming a status code. */
const char* vt_status_string(int status);

/* One-line reason for the latest non-OK status returned on this thread
 * ("" if none).  The pointer stays valid until the next call on the thread. */
const char* vt_last_error(void);

/* Library ABI version (major * 100 + minor). */
int vt_version(void);

/* ------------------------------------------------------------------------
 * Debug builds.  The library can be compiled with VT_CHECKS defined (the
 * build script's checked variant, libvt_gb300_checks.so): every kernel then
 * tests the indices of its index-computed global accesses, skips an access
 * that would fall outside its buffer and records the source line of the
 * first such check.  Nothing traps.  The release build has no checks.
 *
 *   vt_debug_build   1 in a checked build, 0 otherwise.
 *   vt_debug_checks  after the work has finished (it reads device memory
 *                    synchronously): 0 if no check failed since the last
 *                    call, else the source line of a failed check (then
 *                    cleared); -1 if the words could not be read.  Always 0
 *                    in a release build.
 * ------------------------------------------------------------------------ */
int vt_debug_build(void);
int vt_debug_checks(void);

/* vt_selftest_check — one kernel whose bounds check fails by design, to see
 * the debug build's reporting work: it writes buf[i] = i for i = 0 .. n with
 * each write guarded by a check that allows only i < n.  buf (device,
 * uint32[n + 1], 4-byte aligned) holds every index, so nothing lands outside
 * it in either build; a release build writes all n + 1 values, a checked
 * build skips buf[n] and vt_debug_checks() then reports the check's line.
 * 1 <= n <= 2^30.  Argument errors return VT_ERR_INVALID_ARG with nothing
 * launched. */
vt_status vt_selftest_check(uint32_t* buf, int32_t n, void* stream);

/* ------------------------------------------------------------------------
 * vt_workspace_size — workspace bytes of one operation, in one call; the
 * same numbers as the per-operation *_workspace_size functions below.
 *
 *   op  VT_OP_COUNT  (vt_count_tokens):  n = V, the vocabulary size;
 *       VT_OP_SELECT (vt_select_vocab):  n = V;
 *       VT_OP_HEAD   (vt_draft_head, vt_draft_head_ex): M, n = V_high, k;
 *       VT_OP_Q      (vt_draft_q):       M.
 *   Arguments an operation does not use are ignored.  Returns 0 for an
 *   unknown op or sizes out of range.  (vt_draft_head_sets takes per-set
 *   sizes: use vt_draft_head_sets_workspace_size.)
 * ------------------------------------------------------------------------ */
typedef enum {
  VT_OP_COUNT = 0,
  VT_OP_SELECT = 1,
  VT_OP_HEAD = 2,
  VT_OP_Q = 3
} vt_op;
size_t vt_workspace_size(int32_t op, int32_t M, int32_t n, int32_t k);

/* ------------------------------------------------------------------------
 * vt_count_tokens — token-frequency histogram.
 * [VT] Step 1 counts every sampled id into a dict; [FR] Key design counts
 * corpus tokens.  Here the stream is counted into a dense array.
 *
 *   tokens    (device) int32[n], any values; 16-byte aligned.
 *   n         number of tokens, 0 <= n < 2^40.
 *   V         vocabulary size, 1 <= V <= 2^30.
 *   counts    (device) uint32[V]; ACCUMULATED INTO (counts[id] += hits), so
 *             a long stream may be counted in pieces.  Zero it before the
 *             first piece.  Arithmetic is modulo 2^32 per id.
 *   n_invalid (device, nullable) uint64[1]; accumulated: the number of
 *             tokens outside [0, V), which are not counted anywhere.
 *   ws        (device) workspace of vt_count_tokens_workspace_size(V) bytes.
 * ------------------------------------------------------------------------ */
size_t vt_count_tokens_workspace_size(int32_t V);
vt_status vt_count_tokens(const int32_t* tokens, int64_t n, int32_t V,
                          uint32_t* counts, uint64_t* n_invalid, void* ws,
                          size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * vt_select_vocab — top-V_high selection and the two index maps.
 * [VT] Step 2: sort ids by count descending, keep the first V_high; the
 * trimmed index of an id is its rank; coverage = selected / total.
 * Tie rule (the pages leave it to dict order): lower id first, so the
 * result is unique.  Ids with count 0 take part, so exactly V_high ids are
 * always kept.
 *
 *   counts    (device) uint32[V].
 *   V_high    1 <= V_high <= V.
 *   t2f       (device) int32[V_high]: trimmed index -> full id, rank order
 *             (t2f[0] is the most frequent id).
 *   f2t       (device) int32[V]: full id -> trimmed index, -1 if dropped.
 *   sums      (device) uint64[2]: OVERWRITTEN with {kept, total}: the sum of
 *             the kept ids' counts and of all counts.  Coverage is
 *             (double)kept / (double)total, computed by the caller after
 *             the stream is synchronised (NaN when total == 0).
 *   ws        (device) workspace of vt_select_vocab_workspace_size(V) bytes;
 *             no zero-fill needed.  Its 32-bit word at byte 128 is the
 *             call's error word: cleared when the call starts, then 0, or
 *             VT_ERR_TIMEOUT if a look-back wait gave up (t2f, f2t and sums
 *             are then incomplete).
 * ------------------------------------------------------------------------ */
size_t vt_select_vocab_workspace_size(int32_t V);
vt_status vt_select_vocab(const uint32_t* counts, int32_t V, int32_t V_high,
                          int32_t* t2f, int32_t* f2t, uint64_t* sums,
                          void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * vt_gather_rows — reconstruct the trimmed lm_head.
 * [VT] Step 3: W_high = W[trimmed_to_full, :], W stored [vocab, hidden].
 * A bit-exact copy of V_high rows of d bf16 values.
 *
 *   W         (device) bf16[V, d], 16-byte aligned.
 *   d         hidden size, d > 0 and d % 8 == 0.
 *   t2f       (device) int32[V_high].
 *   W_high    (device) bf16[V_high, d], 16-byte aligned, must not overlap W.
 *   n_invalid (device, nullable) uint64[1]; accumulated: rows whose t2f
 *             entry lies outside [0, V); such rows are written as zeros.
 * ------------------------------------------------------------------------ */
vt_status vt_gather_rows(const uint16_t* W, int64_t V, int32_t d,
                         const int32_t* t2f, int32_t V_high, uint16_t* W_high,
                         uint64_t* n_invalid, void* stream);

/* ------------------------------------------------------------------------
 * vt_gather_bias — the kept rows' bias.  [VT] Step 3 copies the old head's
 * bias with the kept ids when the head has one: b_high[i] = b[t2f[i]].
 *
 *   b         (device) float[V], 4-byte aligned.
 *   t2f       (device) int32[V_high].
 *   b_high    (device) float[V_high], must not overlap b.
 *   n_invalid (device, nullable) uint64[1]; accumulated: entries whose t2f
 *             id lies outside [0, V); they are written as 0.
 * ------------------------------------------------------------------------ */
vt_status vt_gather_bias(const float* b, int64_t V, const int32_t* t2f,
                         int32_t V_high, float* b_high, uint64_t* n_invalid,
                         void* stream);

/* ------------------------------------------------------------------------
 * vt_draft_head — one draft step of the trimmed head for M hidden states.
 * [FR] Key design: the draft lm_head projects onto the V_high kept rows only
 * and the softmax is taken over that subset; [VT] Step 4: softmax of the
 * drafter logits, then the chosen trimmed index is mapped back to the full
 * vocabulary through trimmed_to_full before verification.
 *
 *   logit[m][i] = sum_j H[m][j] * W_high[i][j]   (bf16 inputs, fp32 sums)
 *   p[m][i]     = exp(logit[m][i] - max_i) / sum_i exp(logit[m][i] - max_i)
 *   out         = the k largest logits of row m, in descending order;
 *                 out_ids = t2f[i] (full-vocabulary ids), out_probs = p.
 *   Equal logits are ordered by lower full-vocabulary id.
 *
 *   H         (device) bf16, M rows of d values, row stride ldh elements
 *             (ldh >= d, ldh % 8 == 0), 16-byte aligned.
 *   M         number of hidden states (draft-tree nodes), 1 <= M <= 256.
 *   d         hidden size, d % 8 == 0, 8 <= d <= 16384.
 *   W_high    (device) bf16[V_high, d], 16-byte aligned.
 *   V_high    1 <= V_high < 2^31.
 *   t2f       (device, nullable) int32[V_high]; NULL means the identity,
 *             i.e. the untrimmed head over a full vocabulary of V_high rows.
 *   k         1 <= k <= 32 and k <= V_high.  k = 1 is the greedy argmax.
 *   out_ids   (device) int32[M, k].
 *   out_probs (device) float[M, k].
 *   out_logits(device, nullable) float[M, V_high]: every trimmed logit, for
 *             verification; costs an extra write of M*V_high*4 bytes.
 *   ws        (device) workspace of vt_draft_head_workspace_size(M, V_high,
 *             k) bytes.  It must be zero-filled once before its first use;
 *             the counters it holds are left zero by every call.  For
 *             M >= 2 it also holds the [M, V_high] fp32 logits (when
 *             out_logits is NULL).  On every path the 32-bit word at byte
 *             128 is a device error word: 0, or VT_ERR_TIMEOUT if a bounded
 *             wait inside the kernel gave up (readable after a synchronise;
 *             the outputs of that call are then incomplete).  The head never
 *             clears it: a caller that reads a non-zero word writes 0 back.
 *
 * Paths: M = 1 runs a split-V GEMV (CUDA cores, one launch); M >= 2 runs a
 * tcgen05 tensor-core GEMM over all M rows at once plus a per-row softmax
 * and top-k kernel.  One workspace can serve calls of any M.
 * The head's kernels are launched as programmatic dependents of the work
 * ahead of them in the stream: they may become resident while the previous
 * kernel finishes and ask L2 for their first W_high rows meanwhile (a
 * prefetch hint), but read H, t2f, the bias and the workspace, and write
 * anything, only after that kernel has completed; stream order is kept.
 * ------------------------------------------------------------------------ */
size_t vt_draft_head_workspace_size(int32_t M, int32_t V_high, int32_t k);
vt_status vt_draft_head(const uint16_t* H, int32_t M, int32_t d, int64_t ldh,
                        const uint16_t* W_high, int32_t V_high,
                        const int32_t* t2f, int32_t k, int32_t* out_ids,
                        float* out_probs, float* out_logits, void* ws,
                        size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * vt_draft_head_ex — vt_draft_head with options: a bias on the kept rows,
 * a temperature, and drawing from the trimmed distribution instead of
 * taking its top-k.  [VT] Step 3 copies the optional bias of the kept rows
 * with the weight rows (b_high = b[t2f], gathered by the caller); [VT] Step 4
 * draws the draft token from the trimmed softmax with multinomial.  Draws
 * here use the Gumbel-max rule, which draws from the same distribution:
 *
 *   logit[m][i] = sum_j H[m][j] * W_high[i][j] + bias_high[i]
 *   s[m][i]     = logit[m][i] / temperature
 *   p[m][i]     = exp(s[m][i] - max_i s) / sum_i exp(s[m][i] - max_i s)
 *   score       = s                         (VT_HEAD_TOPK)
 *               = s + g(seed, offset, m, t2f[i])   (VT_HEAD_SAMPLE)
 *   out         = the k largest scores of row m, descending (ties: lower
 *                 full id); out_ids = full ids, out_probs = their p,
 *                 out_logits = logit (bias included, before temperature).
 *
 * In VT_HEAD_SAMPLE mode, k = 1 is one draw from p and k > 1 is k draws
 * without replacement.  g is Gumbel noise from the counter-based generator
 * Philox4x32-10 (Salmon et al., SC 2011): x = word 0 of the block at counter
 * (full id, m, offset low 32 bits, offset high 32 bits) and key (seed low,
 * seed high); u = ((x >> 9) + 0.5) / 2^23; g = -log(-log(u)).  Noise is
 * keyed by the full-vocabulary id, so it does not depend on which tokens
 * were kept: whenever the untrimmed head's draw (same seed, offset, m) is a
 * kept token, the trimmed head draws that same token.  Callers advance
 * `offset` once per draft step; m is the hidden state's row in this call.
 *
 *   opts      (host, nullable) options; NULL means no bias, temperature 1,
 *             VT_HEAD_TOPK (exactly vt_draft_head).
 *             bias_high   (device, nullable) float[V_high], 4-byte aligned.
 *             temperature finite and > 0.
 *             mode        VT_HEAD_TOPK or VT_HEAD_SAMPLE.
 *             seed, offset generator key and step counter (sampling only).
 *   Other arguments, the workspace (same size function) and the error word
 *   are those of vt_draft_head; invalid options return VT_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
typedef enum { VT_HEAD_TOPK = 0, VT_HEAD_SAMPLE = 1 } vt_head_mode;

typedef struct {
  const float* bias_high;
  float temperature;
  int32_t mode;
  uint64_t seed;
  uint64_t offset;
} vt_head_options;

vt_status vt_draft_head_ex(const uint16_t* H, int32_t M, int32_t d,
                           int64_t ldh, const uint16_t* W_high,
                           int32_t V_high, const int32_t* t2f, int32_t k,
                           const vt_head_options* opts, int32_t* out_ids,
                           float* out_probs, float* out_logits, void* ws,
                           size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * vt_draft_noise — the Gumbel noise g(seed, offset, m, id) that
 * vt_draft_head_ex adds in VT_HEAD_SAMPLE mode, for n full-vocabulary ids;
 * for verifying draws.  The pages have no counterpart; it is the same
 * device function the sampling kernels call.
 *
 *   full_ids  (device) int32[n];  out (device) float[n];  n >= 0, m >= 0.
 *   Stream-ordered and asynchronous.
 * ------------------------------------------------------------------------ */
vt_status vt_draft_noise(uint64_t seed, uint64_t offset, int32_t m,
                         const int32_t* full_ids, int64_t n, float* out,
                         void* stream);

/* ------------------------------------------------------------------------
 * vt_draft_head_sets — one draft step for hidden states that use different
 * kept vocabularies.  [FR] Limitations: the kept set is one static,
 * corpus-wide vocabulary; vocabularies chosen per domain or per request are
 * future work.  Each set s has its own W_high_sets[s] [V_high_sets[s], d],
 * t2f_sets[s] and optional bias_sets[s], built by the same offline calls
 * from its own token stream; hidden state m is scored against set
 * set_of_row[m] exactly as vt_draft_head_ex would score it alone, and when
 * drawing its noise index is its row m in this call.
 *
 *   H, M (1..256), d, ldh, k, opts, out_ids, out_probs: as vt_draft_head_ex
 *             (opts->bias_high must be NULL: biases are per set).
 *   set_of_row  (host) int32[M], 0 <= set_of_row[m] < S.
 *   W_high_sets (host) array of S device pointers, 16-byte aligned.
 *   V_high_sets (host) int32[S], each >= k.
 *   t2f_sets    (host, nullable) array of S device pointers (entries may
 *               be NULL: identity).
 *   bias_sets   (host, nullable) array of S device pointers (nullable
 *               entries), fp32 [V_high_sets[s]], 4-byte aligned.
 *   ws          (device) vt_draft_head_sets_workspace_size(M, d, k, S,
 *               V_high_sets) bytes, 256-byte aligned, zero-filled once
 *               before its first use.  It begins with the head's workspace,
 *               so its error word is the head's (byte 128).
 * For each set in use: one gather of its rows' hidden states, the head
 * (GEMV for one row, tensor cores for more), one scatter of its outputs.
 * All sets are checked before anything is launched.
 * ------------------------------------------------------------------------ */
size_t vt_draft_head_sets_workspace_size(int32_t M, int32_t d, int32_t k,
                                         int32_t S, const int32_t* V_high_sets);
vt_status vt_draft_head_sets(const uint16_t* H, int32_t M, int32_t d,
                             int64_t ldh, const int32_t* set_of_row, int32_t S,
                             const uint16_t* const* W_high_sets,
                             const int32_t* V_high_sets,
                             const int32_t* const* t2f_sets,
                             const float* const* bias_sets, int32_t k,
                             const vt_head_options* opts, int32_t* out_ids,
                             float* out_probs, void* ws, size_t ws_bytes,
                             void* stream);

/* ------------------------------------------------------------------------
 * vt_draft_q — the full-vocabulary draft distribution of a draft step, for
 * verification.  [FR] Method > Key design: only the draft step is trimmed;
 * the target model verifies with its accept/reject test (rejection
 * sampling), which keeps the output exactly the target's distribution and
 * compares target and draft probabilities over the whole vocabulary, where
 * the trimmed draft gives every dropped id probability 0:
 *
 *   q[m][f] = exp(logits[m][f2t[f]] / T - max) / sum   if f2t[f] >= 0
 *           = 0                                        otherwise,
 *   max, sum over the V_high kept logits of row m (softmax of logit / T).
 *
 *   logits    (device) float[M, V_high], 4-byte aligned: the head's logits
 *             (vt_draft_head / _ex out_logits, bias included).
 *   f2t       (device, nullable) int32[V] from vt_select_vocab; NULL means
 *             the identity (requires V == V_high).
 *   V         full vocabulary size, V >= V_high; 1 <= M <= 65535.
 *   temperature  finite and > 0 (the head's T).
 *   q         (device) float[M, V], 4-byte aligned (16-byte aligned rows
 *             and V % 4 == 0 take the vector path), must not overlap logits.
 *   ws        (device) vt_draft_q_workspace_size(M) bytes, 8-byte aligned;
 *             holds per-row (max, sum); no zero-fill needed.
 * ------------------------------------------------------------------------ */
size_t vt_draft_q_workspace_size(int32_t M);
vt_status vt_draft_q(const float* logits, int32_t M, int32_t V_high,
                     const int32_t* f2t, int32_t V, float temperature,
                     float* q, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * vt_selftest_wait_timeout — runs the library's bounded device wait until it
 * gives up, to check the failure path.  The pages have no counterpart.
 *
 * Every wait of the library's kernels on an mbarrier is bounded by a cycle
 * budget (about a second); when it runs out the kernel writes
 * VT_ERR_TIMEOUT to its error word (byte 128 of the head workspace), stops
 * issuing work and returns, and the context stays usable.  This call
 * launches one 32-thread CTA that waits on an mbarrier nothing arrives on,
 * with the given budget, then writes VT_ERR_TIMEOUT to *err_word.
 *
 *   err_word      (device) uint32, 4-byte aligned; set to VT_ERR_TIMEOUT.
 *   budget_cycles 1 .. 2^31 SM clock cycles (2e6 is about a millisecond).
 * Argument errors return VT_ERR_INVALID_ARG with nothing launched.
 * ------------------------------------------------------------------------ */
vt_status vt_selftest_wait_timeout(uint32_t* err_word, int64_t budget_cycles,
                                   void* stream);

/* ------------------------------------------------------------------------
 * vt_host_step_* — draft steps from host memory, each one CUDA-graph launch.
 * The pages have no counterpart; this serves callers whose hidden states
 * live on the host.  The handle owns a stream, pinned staging buffers,
 * device buffers, a zero-filled head workspace and a CUDA graph of: copy of
 * the staged H [M, d] to the device, then vt_draft_head_ex writing the ids
 * and probabilities straight into a pinned host buffer (device-addressable;
 * no copy node follows).
 *
 *   vt_host_step_create: W_high, V_high, d, t2f, M (1..256), k and opts are
 *     fixed for the handle's life (W_high and t2f must stay valid); opts may
 *     set a bias and a temperature, not VT_HEAD_SAMPLE (a replayed graph
 *     would repeat its step counter).  Runs one step eagerly, then captures.
 *     This call allocates and synchronises; the run call does neither.
 *   vt_host_step_run: copies H_host (host, bf16 [M, d]; skipped when it is
 *     the staging buffer) into the staging buffer, launches the graph,
 *     waits for the step and writes ids_host [M, k] and probs_host [M, k]
 *     (host).  The graph ends with a small kernel that moves the head's
 *     error word (byte 128 of the handle's workspace) into the pinned output
 *     buffer, clears it, and then publishes the step's sequence number there
 *     behind a system-scope fence; the call waits by polling that number
 *     (a stream synchronise takes over after ~10-50 ms, and its error, if
 *     any, is returned as VT_ERR_CUDA).  The graph's last kernel may still
 *     be exiting when the call returns; the next run queues behind it.  If a
 *     bounded wait inside the head gave up, the call returns VT_ERR_TIMEOUT
 *     and writes nothing.  Not thread-safe per handle.
 *   vt_host_step_staging: the pinned [M, d] staging buffer (write H there to
 *     skip the host copy).
 *   vt_host_step_error_word: the device address of the handle's error word
 *     (uint32), for tools and tests of the failure path.
 *   vt_host_step_destroy: synchronises and frees everything (NULL is a no-op).
 * ------------------------------------------------------------------------ */
typedef struct vt_host_step vt_host_step;
vt_status vt_host_step_create(const uint16_t* W_high, int32_t V_high, int32_t d,
                              const int32_t* t2f, int32_t M, int32_t k,
                              const vt_head_options* opts, vt_host_step** out);
vt_status vt_host_step_run(vt_host_step* h, const uint16_t* H_host,
                           int32_t* ids_host, float* probs_host);
uint16_t* vt_host_step_staging(vt_host_step* h);
uint32_t* vt_host_step_error_word(vt_host_step* h);
void vt_host_step_destroy(vt_host_step* h);

/* ------------------------------------------------------------------------
 * vt_draft_head_noalloc — vt_draft_head for callers that cannot allocate.
 * The pages have no counterpart to this call; it exists for integration.
 *
 * Some callers cannot allocate device memory where they run a draft step
 * (inside a CUDA stream capture that must not gain allocation nodes, on
 * hosts that forbid allocation after start-up, or as a plugin confined to
 * another framework's memory pool), so they cannot provide the workspace
 * vt_draft_head needs.  This call computes what vt_draft_head computes,
 * with the same arguments minus the workspace, and allocates nothing: its
 * scratch is one fixed 1 MiB array in device memory that the library
 * defines and every GPU that loads the library keeps until exit.
 * It always runs the GEMV kernel, four hidden states at a time.  For M = 1
 * that is vt_draft_head's own kernel.  For M >= 2 vt_draft_head uses the
 * tensor-core path, which sums in another order, so the two calls agree
 * within the head's tolerances (logits within 1e-3 * (1 + |logit|),
 * probabilities within 1e-4), and their ids agree except where two
 * candidates' logits are closer than that.
 *
 *   Limit     the GEMV scratch, 2048 + 4096 * min(M, 4) * P bytes with
 *             P = 4 + 2k rounded up to a multiple of 4, must fit in 1 MiB:
 *             any k <= 32 for M <= 3, k <= 28 for M >= 4; larger requests
 *             return VT_ERR_UNSUPPORTED.
 *   Set-up    the first call on each device looks up the array's device
 *             address and zero-fills its counters with a synchronous
 *             cudaMemset; make that first call before any stream capture.
 *   Sharing   all calls on a device share the one array; calls that overlap
 *             on the GPU (unordered streams) race on it and give wrong
 *             results.  Calls on one stream are safe.
 *   Timeouts  the kernel's one bounded wait (the final merge's copy of the
 *             partial results, about a second) cannot be reported by this
 *             call: its error word lies inside the private array and no
 *             call returns it, nor clears it.  When that wait gives up the
 *             call leaves the out_ids rows from the one it failed on
 *             unwritten.  A caller that must detect this fills out_ids with
 *             -1 before the call (no full-vocabulary id is negative) and
 *             checks for -1 after synchronising.
 * ------------------------------------------------------------------------ */
vt_status vt_draft_head_noalloc(const uint16_t* H, int32_t M, int32_t d,
                                int64_t ldh, const uint16_t* W_high,
                                int32_t V_high, const int32_t* t2f, int32_t k,
                                int32_t* out_ids, float* out_probs,
                                float* out_logits, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VT_H_ */
