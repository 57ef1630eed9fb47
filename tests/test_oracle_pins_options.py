"""Pins of the oracle's head options, checked against things other than the
oracle itself: the published known-answer vectors of the Philox4x32-10
generator, the Gumbel-max law (the drawn ids follow softmax(l / T), and the
k best of l / T + noise follow the law of draws without replacement),
closed forms for the bias and the temperature, and invariants of the noise
(it is keyed by full-vocabulary id, so trimming or reordering the kept rows
never changes a kept token's draw).  All on the CPU."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import synth

MASK = 0xFFFFFFFF

# Known-answer vectors of Philox4x32-10 published with the generator
# (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011, and
# its reference distribution): counter, key -> output block.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((MASK, MASK, MASK, MASK), (MASK, MASK),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def bf16(a) -> np.ndarray:
    return synth.bf16_bits(torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def one_hot_head(values, rows=1, d=8):
    """Hidden states e_0 against a weight whose column 0 holds `values`
    (bf16-exact): every logit is exactly the matching value."""
    V_high = len(values)
    W = np.zeros((V_high, d), np.float32)
    W[:, 0] = values
    H = np.zeros((rows, d), np.float32)
    H[:, 0] = 1.0
    return bf16(H), bf16(W)


def softmax(x):
    e = np.exp(x - np.max(x))
    return e / e.sum()


def test_philox_known_answers(oracle_lib):
    for ctr, key, want in PHILOX_KAT:
        assert oracle.philox4x32_10(ctr, key).tolist() == list(want)


def test_gumbel_noise_is_standard_gumbel(oracle_lib):
    """200000 noise values of distinct ids: Kolmogorov-Smirnov against the
    standard Gumbel law, and its mean (Euler's constant) and variance
    (pi^2 / 6)."""
    g = oracle.gumbel_noise(12345, 7, 3, np.arange(200_000))
    assert stats.kstest(g, stats.gumbel_r.cdf).pvalue > 1e-4
    assert abs(g.mean() - np.euler_gamma) < 0.01
    assert abs(g.var() - np.pi ** 2 / 6) < 0.03


@pytest.mark.parametrize("temperature,use_bias", [(1.0, False), (0.5, True),
                                                  (2.0, False)])
def test_gumbel_max_draws_follow_softmax(oracle_lib, temperature, use_bias):
    """One draw per hidden state (each state has its own noise): over 100000
    states the ids follow softmax((l + b) / T) (chi-square)."""
    values = np.array([0.5, 1.0, -0.25, 2.0, 0.0, 1.5, -1.0, 0.75])
    bias = (np.array([0.1, -0.2, 0.3, 0.0, -0.5, 0.25, 0.4, -0.1], np.float32)
            if use_bias else None)
    N = 100_000
    H, W = one_hot_head(values, rows=N)
    r = oracle.draft_head_ex(H, W, None, 1, bias=bias, temperature=temperature,
                             sample=True, seed=2024, offset=11)
    counts = np.bincount(r["ids"][:, 0], minlength=values.size)
    lb = values + (bias.astype(np.float64) if use_bias else 0.0)
    p = softmax(lb / temperature)
    assert stats.chisquare(counts, N * p).pvalue > 1e-4
    # the reported probability is that of the drawn token
    np.testing.assert_allclose(r["probs"][:, 0], p[r["ids"][:, 0]], rtol=1e-12)


def test_gumbel_topk_is_draws_without_replacement(oracle_lib):
    """k = 2 over four tokens: ordered pairs (i, j) appear with probability
    p_i * p_j / (1 - p_i) (chi-square over the 12 pairs)."""
    values = np.array([1.0, 0.0, -0.5, 0.5])
    N = 120_000
    H, W = one_hot_head(values, rows=N)
    r = oracle.draft_head_ex(H, W, None, 2, sample=True, seed=99, offset=0)
    p = softmax(values)
    pairs = r["ids"][:, 0] * 4 + r["ids"][:, 1]
    counts = np.bincount(pairs, minlength=16)
    expect = np.array([p[i] * p[j] / (1 - p[i]) if i != j else 0.0
                       for i in range(4) for j in range(4)])
    keep = expect > 0
    assert counts[~keep].sum() == 0
    assert stats.chisquare(counts[keep], N * expect[keep]).pvalue > 1e-4


def test_defaults_equal_the_plain_head(oracle_lib):
    H = synth.bf16_bits(synth.normal_bf16((5, 64), 1.0, seed=1))
    W = synth.bf16_bits(synth.normal_bf16((300, 64), 0.05, seed=2))
    t2f = synth.rank_permutation(600, 3)[:300].numpy()
    a = oracle.draft_head(H, W, t2f, 7)
    b = oracle.draft_head_ex(H, W, t2f, 7)
    for key in ("ids", "probs", "logits", "trimmed", "row_max", "row_sumexp"):
        assert np.array_equal(a[key], b[key]), key


def test_bias_and_temperature_closed_forms(oracle_lib):
    """Logits are H.W^T + b (numpy fp64 matmul); probabilities are
    softmax((H.W^T + b) / T) over all kept rows (scipy), top-k ids do not
    depend on T."""
    M, d, V_high = 3, 48, 200
    H = synth.normal_bf16((M, d), 1.0, seed=4)
    W = synth.normal_bf16((V_high, d), 0.05, seed=5)
    b = np.random.default_rng(6).normal(0, 0.3, V_high).astype(np.float32)
    Hh, Wh = synth.bf16_bits(H), synth.bf16_bits(W)
    ref_logits = H.double().numpy() @ W.double().numpy().T + b.astype(np.float64)
    for T in (1.0, 0.7, 3.0):
        r = oracle.draft_head_ex(Hh, Wh, None, V_high, bias=b, temperature=T)
        for m in range(M):
            idx = r["trimmed"][m]
            np.testing.assert_allclose(r["logits"][m], ref_logits[m, idx],
                                       rtol=1e-12, atol=1e-12)
            from scipy.special import softmax as sp_softmax
            np.testing.assert_allclose(r["probs"][m],
                                       sp_softmax(ref_logits[m] / T)[idx],
                                       rtol=1e-10)
        t1 = oracle.draft_head_ex(Hh, Wh, None, 10, bias=b, temperature=1.0)
        assert np.array_equal(r["ids"][:, :10], t1["ids"])


def test_noise_is_keyed_by_full_id(oracle_lib):
    """Reordering the kept rows (and t2f with them) changes no draw: the
    noise belongs to the token, not to its trimmed position."""
    M, d, V_high = 40, 32, 120
    Hh = synth.bf16_bits(synth.normal_bf16((M, d), 1.0, seed=7))
    Wh = synth.bf16_bits(synth.normal_bf16((V_high, d), 0.2, seed=8))
    t2f = synth.rank_permutation(1000, 9)[:V_high].numpy()
    perm = np.random.default_rng(10).permutation(V_high)
    a = oracle.draft_head_ex(Hh, Wh, t2f, 3, sample=True, seed=5, offset=77)
    b = oracle.draft_head_ex(Hh, np.ascontiguousarray(Wh[perm]), t2f[perm], 3,
                             sample=True, seed=5, offset=77)
    assert np.array_equal(a["ids"], b["ids"])
    np.testing.assert_array_equal(a["scores"], b["scores"])


def test_trimmed_draw_equals_untrimmed_draw_when_kept(oracle_lib):
    """Same seed and step: whenever the untrimmed head's draw is a kept
    token, the trimmed head draws that same token (the maximum of
    l / T + g over a subset containing the overall maximiser is that
    maximiser)."""
    M, d, V = 400, 32, 256
    Hh = synth.bf16_bits(synth.normal_bf16((M, d), 1.0, seed=11))
    Wf = synth.bf16_bits(synth.normal_bf16((V, d), 0.3, seed=12))
    t2f = np.sort(np.random.default_rng(13).permutation(V)[:128]).astype(np.int32)
    full = oracle.draft_head_ex(Hh, Wf, None, 1, sample=True, seed=3,
                                offset=5, temperature=0.8)
    trim = oracle.draft_head_ex(Hh, np.ascontiguousarray(Wf[t2f]), t2f, 1,
                                sample=True, seed=3, offset=5, temperature=0.8)
    kept = np.isin(full["ids"][:, 0], t2f)
    assert kept.sum() > 100
    assert np.array_equal(full["ids"][kept, 0], trim["ids"][kept, 0])


def philox_gumbel(seed, offset, m, full_id):
    """Gumbel noise of one token built from the generator's block alone
    (the block is pinned by the published known-answer vectors): counter
    (full id, hidden state, offset low word, offset high word), key (seed
    low word, seed high word); u from the top 23 bits of word 0 at the
    middle of its cell; g = -log(-log(u))."""
    x = oracle.philox4x32_10(
        (full_id, m, offset & MASK, offset >> 32), (seed & MASK, seed >> 32))[0]
    u = ((int(x) >> 9) + 0.5) / 2.0 ** 23
    return -np.log(-np.log(u))


def test_sampled_rows_are_keyed_by_their_row_in_the_batch(oracle_lib):
    """[VT] Step 4 draws one token per hidden state; the draw of hidden state
    m uses noise index m, its row in the caller's batch.  A call over a
    slice of the batch that starts at row j (m_base = j) must draw exactly
    what those rows draw in the whole batch, and every drawn token's score
    must be its s plus the generator's noise for its row and full id."""
    M, d, V_high, k = 7, 32, 300, 4
    seed, offset = (0x1234_5678_9ABC, (3 << 32) + 17)
    Hh = synth.bf16_bits(synth.normal_bf16((M, d), 1.0, seed=31))
    Wh = synth.bf16_bits(synth.normal_bf16((V_high, d), 0.2, seed=32))
    t2f = synth.rank_permutation(900, 33)[:V_high].numpy()
    whole = oracle.draft_head_ex(Hh, Wh, t2f, k, sample=True, seed=seed,
                                 offset=offset, temperature=0.7)
    for j, n in ((0, 1), (1, 2), (4, 3), (6, 1)):
        part = oracle.draft_head_ex(np.ascontiguousarray(Hh[j:j + n]), Wh, t2f,
                                    k, sample=True, seed=seed, offset=offset,
                                    temperature=0.7, m_base=j)
        assert np.array_equal(part["ids"], whole["ids"][j:j + n]), j
        np.testing.assert_array_equal(part["scores"], whole["scores"][j:j + n])
    g = whole["scores"] - whole["logits"] / 0.7
    for m in range(M):
        want = [philox_gumbel(seed, offset, m, int(f)) for f in whole["ids"][m]]
        np.testing.assert_allclose(g[m], want, rtol=0, atol=1e-9)


def test_steps_and_seeds_change_the_draw(oracle_lib):
    """Different offsets (steps) or seeds give different noise; the same
    (seed, offset) repeats it."""
    ids = np.arange(1000)
    a = oracle.gumbel_noise(1, 0, 0, ids)
    assert np.array_equal(a, oracle.gumbel_noise(1, 0, 0, ids))
    for other in (oracle.gumbel_noise(1, 1, 0, ids),
                  oracle.gumbel_noise(2, 0, 0, ids),
                  oracle.gumbel_noise(1, 1 << 32, 0, ids),
                  oracle.gumbel_noise(1 << 32, 0, 0, ids),
                  oracle.gumbel_noise(1, 0, 1, ids)):
        assert abs(np.corrcoef(a, other)[0, 1]) < 0.1


def test_bias_gather_vs_fancy_index(oracle_lib):
    """b_high = b[t2f] (numpy fancy indexing); out-of-range ids give 0 and
    are counted."""
    rng = np.random.default_rng(21)
    b = rng.normal(0, 1, 500).astype(np.float32)
    t2f = rng.permutation(500)[:123].astype(np.int32)
    out, bad = oracle.gather_bias(b, t2f)
    assert bad == 0 and np.array_equal(out, b[t2f])
    t2f[[3, 50]] = [-1, 500]
    out, bad = oracle.gather_bias(b, t2f)
    assert bad == 2 and out[3] == 0 and out[50] == 0
    keep = np.ones(123, bool)
    keep[[3, 50]] = False
    assert np.array_equal(out[keep], b[t2f[keep]])


def test_draft_q_closed_form(oracle_lib):
    """q is scipy's softmax((H.W^T + b) / T) over the kept rows placed at the
    kept ids (numpy fancy indexing), exactly 0 elsewhere, and sums to 1."""
    from scipy.special import softmax as sp_softmax
    M, d, V, V_high = 4, 40, 700, 230
    H = synth.normal_bf16((M, d), 1.0, seed=31)
    W = synth.normal_bf16((V_high, d), 0.1, seed=32)
    b = np.random.default_rng(33).normal(0, 0.2, V_high).astype(np.float32)
    t2f = synth.rank_permutation(V, 34)[:V_high].numpy()
    logits = H.double().numpy() @ W.double().numpy().T + b.astype(np.float64)
    for T in (1.0, 0.6):
        q = oracle.draft_q(synth.bf16_bits(H), synth.bf16_bits(W), t2f, V,
                           bias=b, temperature=T)
        want = np.zeros((M, V))
        want[:, t2f] = sp_softmax(logits / T, axis=1)
        np.testing.assert_allclose(q, want, rtol=1e-12, atol=1e-15)
        dropped = np.setdiff1d(np.arange(V), t2f)
        assert np.all(q[:, dropped] == 0.0)
        for m in range(M):
            assert abs(math_fsum(q[m]) - 1.0) < 1e-12


def test_draft_q_untrimmed_and_drawn_probabilities(oracle_lib):
    """With the identity map q is the full softmax; the probability the head
    reports for a drawn token is q at that token."""
    from scipy.special import softmax as sp_softmax
    M, d, V = 3, 32, 300
    H = synth.normal_bf16((M, d), 1.0, seed=41)
    W = synth.normal_bf16((V, d), 0.2, seed=42)
    q = oracle.draft_q(synth.bf16_bits(H), synth.bf16_bits(W), None, V,
                       temperature=0.9)
    np.testing.assert_allclose(
        q, sp_softmax((H.double().numpy() @ W.double().numpy().T) / 0.9, axis=1),
        rtol=1e-12)
    r = oracle.draft_head_ex(synth.bf16_bits(H), synth.bf16_bits(W), None, 4,
                             temperature=0.9, sample=True, seed=1, offset=2)
    for m in range(M):
        np.testing.assert_allclose(r["probs"][m], q[m, r["ids"][m]], rtol=1e-12)


def math_fsum(x):
    import math
    return math.fsum(float(v) for v in x)
