"""Pins for the CPU oracle, against things other than the oracle itself.

Each pin comes from the pages (hand-worked fixtures under tests/golden/ that
restate the pages' steps on a case small enough to do by hand), a library
routine that the step reduces to in a special case (numpy.bincount,
numpy.lexsort, numpy fp64 matmul, scipy softmax), a closed form (Zipf
coverage, unit-vector hidden state, uniform logits), an invariant the pages
imply (maps are inverse, trimmed logits equal the full head at kept ids), or
brute force written as a different algorithm on tiny inputs (Counter,
selection by repeated maximum, exactly rounded sums).  Together they catch a
dropped term, a wrong sign, a wrong index or a transposed operand anywhere in
the oracle.
"""
import collections
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import golden_io
import synth


def bf16(values) -> np.ndarray:
    """float values -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------- fixtures

def test_golden_vocab_build(oracle_lib):
    rec = golden_io.read("vocab_build_worked.txt")
    V = int(golden_io.first(rec, "V")[0])
    tokens = np.array([int(x) for x in golden_io.first(rec, "tokens")], np.int32)
    counts, n_invalid = oracle_lib.count_tokens(tokens, V)
    assert counts.tolist() == [int(x) for x in golden_io.first(rec, "counts")]
    assert n_invalid == int(golden_io.first(rec, "n_invalid")[0])
    full = oracle_lib.select_vocab(counts, V)
    assert full["t2f"].tolist() == [int(x) for x in golden_io.first(rec, "order")]
    assert full["total"] == int(golden_io.first(rec, "total")[0])
    selects = collections.defaultdict(dict)
    for vals in golden_io.all_of(rec, "select"):
        vh, key, rest = int(vals[0]), vals[1], vals[2:]
        selects[vh][key] = rest
    assert len(selects) == 2
    for vh, exp in selects.items():
        r = oracle_lib.select_vocab(counts, vh)
        assert r["t2f"].tolist() == [int(x) for x in exp["t2f"]]
        assert r["f2t"].tolist() == [int(x) for x in exp["f2t"]]
        assert r["kept"] == int(exp["kept"][0])
        assert exp["kept"][1] == "coverage"
        assert r["coverage"] == float(exp["kept"][2])


def _load_head_fixture(name):
    rec = golden_io.read(name)
    d = int(golden_io.first(rec, "d")[0])
    t2f = np.array([int(x) for x in golden_io.first(rec, "t2f")], np.int32)
    H = bf16([[float(x) for x in golden_io.first(rec, "H")]])
    W = bf16([[float(x) for x in row] for row in golden_io.all_of(rec, "W")])
    assert H.shape == (1, d) and W.shape == (t2f.size, d)
    return rec, H, W, t2f


def test_golden_draft_head(oracle_lib):
    rec, H, W, t2f = _load_head_fixture("draft_head_worked.txt")
    logits = oracle_lib.head_logits(H, W)[0]
    assert logits.tolist() == [float(x) for x in golden_io.first(rec, "logits")]
    k = int(golden_io.first(rec, "k")[0])
    r = oracle_lib.draft_head(H, W, t2f, k)
    assert r["trimmed"][0].tolist() == [int(x) for x in golden_io.first(rec, "top_trimmed")]
    assert r["ids"][0].tolist() == [int(x) for x in golden_io.first(rec, "top_ids")]
    probs = [float(x) for x in golden_io.first(rec, "probs")]
    for j, t in enumerate(r["trimmed"][0]):
        assert r["probs"][0, j] == pytest.approx(probs[t], rel=1e-14, abs=0)
    # all four probabilities (k = V_high) sum to one
    r4 = oracle_lib.draft_head(H, W, t2f, 4)
    assert math.fsum(r4["probs"][0]) == pytest.approx(1.0, abs=1e-15)


def test_golden_topk_ties(oracle_lib):
    rec, H, W, t2f = _load_head_fixture("topk_ties_worked.txt")
    k = int(golden_io.first(rec, "k")[0])
    r = oracle_lib.draft_head(H, W, t2f, k)
    assert r["ids"][0].tolist() == [int(x) for x in golden_io.first(rec, "top_ids")]
    assert r["trimmed"][0].tolist() == [int(x) for x in golden_io.first(rec, "top_trimmed")]
    assert np.all(r["probs"] == float(golden_io.first(rec, "probs_each")[0]))


# ---------------------------------------------------------------- histogram

@pytest.mark.parametrize("V,n,seed", [(7, 0, 0), (7, 50, 1), (100, 5000, 2),
                                      (4096, 200_000, 3)])
def test_histogram_vs_bincount(oracle_lib, V, n, seed):
    rng = np.random.default_rng(seed)
    tokens = rng.integers(-3, V + 3, size=n, dtype=np.int64).astype(np.int32)
    counts, n_invalid = oracle_lib.count_tokens(tokens, V)
    valid = tokens[(tokens >= 0) & (tokens < V)]
    assert np.array_equal(counts, np.bincount(valid, minlength=V).astype(np.uint64))
    assert n_invalid == n - valid.size
    assert int(counts.sum()) == n - n_invalid


def test_histogram_brute_force_counter(oracle_lib):
    tokens = synth.zipf_tokens(3000, 64, 1.1, seed=11).numpy()
    counts, _ = oracle_lib.count_tokens(tokens, 64)
    c = collections.Counter(tokens.tolist())
    assert [c.get(i, 0) for i in range(64)] == counts.tolist()


# ---------------------------------------------------------------- selection

def _brute_select(counts, V_high):
    """Selection by repeated maximum: take the most frequent remaining id,
    lowest id on ties, V_high times."""
    remaining = list(range(len(counts)))
    chosen = []
    for _ in range(V_high):
        best = remaining[0]
        for i in remaining[1:]:
            if counts[i] > counts[best]:
                best = i
        chosen.append(best)
        remaining.remove(best)
    return chosen


@pytest.mark.parametrize("V,V_high,maxc,seed", [(1, 1, 3, 0), (12, 5, 3, 1),
                                               (40, 40, 2, 2), (64, 17, 1000, 3),
                                               (64, 1, 0, 4)])
def test_select_brute_force(oracle_lib, V, V_high, maxc, seed):
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, maxc + 1, size=V).astype(np.uint64)
    r = oracle_lib.select_vocab(counts, V_high)
    assert r["t2f"].tolist() == _brute_select(counts.tolist(), V_high)


@pytest.mark.parametrize("V,V_high,seed", [(4096, 1024, 5), (5000, 4999, 6),
                                           (128256, 32768, 7)])
def test_select_vs_lexsort_and_invariants(oracle_lib, V, V_high, seed):
    rng = np.random.default_rng(seed)
    # heavy ties: small count range
    counts = rng.integers(0, 50, size=V).astype(np.uint64)
    r = oracle_lib.select_vocab(counts, V_high)
    order = np.lexsort((np.arange(V), -counts.astype(np.int64)))
    assert np.array_equal(r["t2f"], order[:V_high].astype(np.int32))
    t2f, f2t = r["t2f"], r["f2t"]
    # exactly V_high distinct kept ids, V - V_high dropped
    assert len(set(t2f.tolist())) == V_high
    assert int((f2t == -1).sum()) == V - V_high
    # maps are mutual inverses on the kept set
    assert np.array_equal(f2t[t2f], np.arange(V_high, dtype=np.int32))
    kept_mask = f2t >= 0
    assert np.array_equal(t2f[f2t[kept_mask]], np.nonzero(kept_mask)[0])
    # min kept key beats max dropped key; key strictly decreasing along t2f
    key = counts.astype(np.int64) * (V + 1) + (V - np.arange(V))
    assert np.all(np.diff(key[t2f]) < 0)
    if V_high < V:
        assert key[t2f].min() > key[~kept_mask].max()
    assert r["kept"] == int(counts[t2f].sum())
    assert r["total"] == int(counts.sum())


def test_select_full_sort_special_case(oracle_lib):
    counts = np.array([5, 9, 5, 0, 9, 1], dtype=np.uint64)
    r = oracle_lib.select_vocab(counts, 6)
    assert r["t2f"].tolist() == [1, 4, 0, 2, 5, 3]
    assert r["coverage"] == 1.0


def test_coverage_exact_rational(oracle_lib):
    rng = np.random.default_rng(9)
    counts = rng.integers(0, 10**9, size=1000).astype(np.uint64)
    r = oracle_lib.select_vocab(counts, 300)
    frac = Fraction(int(np.sort(counts)[::-1][:300].sum()), int(counts.sum()))
    assert r["coverage"] == float(frac)  # one correctly rounded division


def test_coverage_zero_total_is_nan(oracle_lib):
    r = oracle_lib.select_vocab(np.zeros(8, np.uint64), 3)
    assert r["t2f"].tolist() == [0, 1, 2]
    assert math.isnan(r["coverage"])


def test_coverage_zipf_closed_form(oracle_lib):
    """Expected coverage of the top V_high ranks of Zipf(s) over V is
    H_{V_high}(s) / H_V(s); a 1e6-token draw sits within a few standard
    errors of it."""
    V, V_high, s, n = 4096, 1024, 1.1, 1_000_000
    tokens = synth.zipf_tokens(n, V, s, seed=1001).numpy()
    counts, _ = oracle_lib.count_tokens(tokens, V)
    r = oracle_lib.select_vocab(counts, V_high)
    Hs = lambda m: math.fsum(j ** -s for j in range(1, m + 1))
    expect = Hs(V_high) / Hs(V)
    sigma = math.sqrt(expect * (1 - expect) / n)
    # the selected set is the empirical top, which can only beat the
    # expected-rank set; allow 6 sigma either way
    assert abs(r["coverage"] - expect) < 6 * sigma + 2e-3


# ------------------------------------------------------------------- gather

def test_gather_vs_fancy_index(oracle_lib):
    rng = np.random.default_rng(3)
    W = rng.integers(0, 1 << 16, size=(300, 24), dtype=np.uint32).astype(np.uint16)
    t2f = rng.permutation(300)[:77].astype(np.int32)
    out, rc = oracle_lib.gather_rows(W, t2f)
    assert rc == 0
    assert np.array_equal(out, W[t2f])


def test_gather_invalid_rows_zero(oracle_lib):
    W = np.arange(40, dtype=np.uint16).reshape(5, 8) + 1
    out, rc = oracle_lib.gather_rows(W, np.array([4, -1, 5, 0], np.int32))
    assert rc == 2
    assert np.array_equal(out[0], W[4]) and np.array_equal(out[3], W[0])
    assert not out[1].any() and not out[2].any()


# --------------------------------------------------------------------- head

def _rand_head(rng, M, d, V_high, hs=1.0, ws=0.02):
    H = bf16(rng.normal(0, hs, size=(M, d)))
    W = bf16(rng.normal(0, ws, size=(V_high, d)))
    return H, W


def test_head_unit_vector_picks_column(oracle_lib):
    rng = np.random.default_rng(1)
    _, W = _rand_head(rng, 1, 32, 50)
    for j in (0, 7, 31):
        H = np.zeros((1, 32), np.uint16)
        H[0, j] = bf16([1.0])[0]
        assert np.array_equal(oracle_lib.head_logits(H, W)[0], bf16_to_f64(W[:, j]))


def test_head_logits_vs_numpy_matmul(oracle_lib):
    rng = np.random.default_rng(2)
    H, W = _rand_head(rng, 3, 256, 300)
    got = oracle_lib.head_logits(H, W)
    ref = bf16_to_f64(H) @ bf16_to_f64(W).T
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_head_brute_force_tiny(oracle_lib):
    """Exactly rounded sums, exp and selection by repeated maximum."""
    rng = np.random.default_rng(4)
    M, d, V_high, k = 2, 16, 9, 4
    H, W = _rand_head(rng, M, d, V_high, ws=1.0)
    t2f = rng.permutation(40)[:V_high].astype(np.int32)
    r = oracle_lib.draft_head(H, W, t2f, k)
    Hf, Wf = bf16_to_f64(H), bf16_to_f64(W)
    for m in range(M):
        lg = [math.fsum(Hf[m, j] * Wf[i, j] for j in range(d)) for i in range(V_high)]
        mx = max(lg)
        z = math.fsum(math.exp(x - mx) for x in lg)
        left = list(range(V_high))
        for rank in range(k):
            best = left[0]
            for i in left[1:]:
                if lg[i] > lg[best] or (lg[i] == lg[best] and t2f[i] < t2f[best]):
                    best = i
            left.remove(best)
            assert r["trimmed"][m, rank] == best
            assert r["ids"][m, rank] == t2f[best]
            assert r["logits"][m, rank] == pytest.approx(lg[best], rel=1e-13, abs=1e-13)
            assert r["probs"][m, rank] == pytest.approx(math.exp(lg[best] - mx) / z, rel=1e-12)
        assert r["row_max"][m] == pytest.approx(mx, rel=1e-13)


def test_head_identity_vs_scipy_softmax(oracle_lib):
    """V_high = V with the identity map is the untrimmed head: the library
    softmax of the numpy fp64 logits, ordered by numpy's stable argsort."""
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    H, W = _rand_head(rng, 2, 64, 500, ws=0.3)
    k = 12
    r = oracle_lib.draft_head(H, W, None, k)
    lg = bf16_to_f64(H) @ bf16_to_f64(W).T
    p = scipy_special.softmax(lg, axis=1)
    for m in range(2):
        top = np.argsort(-lg[m], kind="stable")[:k]
        assert r["ids"][m].tolist() == top.tolist()
        np.testing.assert_allclose(r["probs"][m], p[m, top], rtol=1e-11)


def test_head_softmax_invariants(oracle_lib):
    rng = np.random.default_rng(6)
    H, W = _rand_head(rng, 1, 128, 200, ws=0.2)
    r = oracle_lib.draft_head(H, W, None, 200)  # k = V_high: every probability
    p, lg = r["probs"][0], r["logits"][0]
    assert math.fsum(p) == pytest.approx(1.0, abs=1e-12)
    assert np.all(np.diff(lg) <= 0) and np.all(np.diff(p) <= 0)
    i, j = 3, 150
    assert p[i] / p[j] == pytest.approx(math.exp(lg[i] - lg[j]), rel=1e-12)
    assert r["row_sumexp"][0] == pytest.approx(1.0 / p[0], rel=1e-12)


def test_head_uniform_logits(oracle_lib):
    W = np.zeros((37, 16), np.uint16)
    H = bf16(np.ones((1, 16)))
    r = oracle_lib.draft_head(H, W, None, 5)
    assert r["ids"][0].tolist() == [0, 1, 2, 3, 4]
    np.testing.assert_allclose(r["probs"][0], 1.0 / 37, rtol=1e-15)


def test_head_large_logits_no_overflow(oracle_lib):
    """Logits in the thousands: exp(l) overflows, exp(l - max) does not."""
    rng = np.random.default_rng(7)
    H = bf16(rng.normal(0, 64.0, size=(1, 256)))
    W = bf16(rng.normal(0, 1.0, size=(100, 256)))
    r = oracle_lib.draft_head(H, W, None, 100)
    assert np.all(np.isfinite(r["probs"]))
    assert abs(r["logits"][0, 0]) > 700
    assert math.fsum(r["probs"][0]) == pytest.approx(1.0, abs=1e-12)


def test_trimmed_equals_full_at_kept_ids(oracle_lib):
    """The trimmed head equals the full head restricted to the kept rows,
    and the trimmed argmax equals the full argmax whenever that id is kept."""
    rng = np.random.default_rng(8)
    V, V_high, d = 600, 150, 64
    H, W = _rand_head(rng, 4, d, V, ws=0.5)
    counts = rng.integers(0, 30, size=V).astype(np.uint64)
    sel = oracle_lib.select_vocab(counts, V_high)
    W_high, rc = oracle_lib.gather_rows(W, sel["t2f"])
    assert rc == 0
    full = oracle_lib.head_logits(H, W)
    trim = oracle_lib.head_logits(H, W_high)
    assert np.array_equal(trim, full[:, sel["t2f"]])
    rf = oracle_lib.draft_head(H, W, None, 1)
    rt = oracle_lib.draft_head(H, W_high, sel["t2f"], 1)
    n_kept_argmax = 0
    for m in range(4):
        if sel["f2t"][rf["ids"][m, 0]] >= 0:
            n_kept_argmax += 1
            assert rt["ids"][m, 0] == rf["ids"][m, 0]
            # same numerator, fewer terms in the denominator
            assert rt["probs"][m, 0] >= rf["probs"][m, 0]
    # force the case at least once: keep the full argmax of row 0
    counts[rf["ids"][0, 0]] = 10**6
    sel = oracle_lib.select_vocab(counts, V_high)
    W_high, _ = oracle_lib.gather_rows(W, sel["t2f"])
    rt = oracle_lib.draft_head(H, W_high, sel["t2f"], 1)
    assert rt["ids"][0, 0] == rf["ids"][0, 0]
    assert sel["t2f"][0] == rf["ids"][0, 0]
