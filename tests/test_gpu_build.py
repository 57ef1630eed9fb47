"""GPU parity of the offline build: histogram, selection + maps + sums, and
row gather, against the CPU oracle, bit-exact, through the C ABI."""
import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import bits_host, need_cuda, u32_host

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ count

def _count_and_compare(tokens_host: np.ndarray, V: int):
    dev = need_cuda()
    tokens = torch.from_numpy(tokens_host).to(dev)
    counts, n_invalid = vt.count_tokens(tokens, V)
    got = u32_host(counts)
    ref, ref_invalid = oracle.count_tokens(tokens_host, V)
    assert np.array_equal(got.astype(np.uint64), ref)
    assert int(n_invalid.item()) == ref_invalid
    return got


def test_count_tiny_zipf():
    cfg = synth.TINY_BUILD
    tokens = synth.zipf_tokens(cfg.n_tokens, cfg.V, cfg.s, cfg.seed).numpy()
    _count_and_compare(tokens, cfg.V)


@pytest.mark.parametrize("n", [0, 1, 3, 5, 4097, 1_000_003])
def test_count_ragged_with_invalid_ids(n):
    rng = np.random.default_rng(n)
    V = 5000
    tokens = rng.integers(-20, V + 20, size=n).astype(np.int32)
    if n:
        tokens[0] = np.iinfo(np.int32).min
        tokens[-1] = np.iinfo(np.int32).max
    _count_and_compare(tokens, V)


def test_count_byte_wrap_carry_chains():
    """Four ids share one shared-memory word; millions of hits make every
    byte wrap thousands of times with carry chains through the word."""
    rng = np.random.default_rng(42)
    tokens = rng.choice(4, size=6_000_000, p=[0.4, 0.3, 0.2, 0.1]).astype(np.int32)
    got = _count_and_compare(tokens, 8)
    assert got[4:].sum() == 0


@pytest.mark.parametrize("V", [4096, 4097])
def test_count_mostly_invalid_ids(V):
    """Nine tokens in ten out of range: the invalid count (kept in a padding
    byte past the histogram when V % 4 == 0) wraps thousands of times per CTA
    and must still be exact, and no valid count may move."""
    rng = np.random.default_rng(V)
    n = 3_000_017
    tokens = rng.integers(0, V, size=n).astype(np.int32)
    bad = rng.random(n) < 0.9
    tokens[bad] = rng.choice(np.array([-1, V, V + 3, np.iinfo(np.int32).min,
                                       np.iinfo(np.int32).max], dtype=np.int32),
                             size=int(bad.sum()))
    _count_and_compare(tokens, V)


def test_count_single_hot_id():
    tokens = np.full(3_000_001, 7, dtype=np.int32)
    got = _count_and_compare(tokens, 10)
    assert got[7] == 3_000_001


def test_count_multi_pass_large_vocab():
    """V above the per-pass shared-memory budget: counted in two passes."""
    V = 300_000
    tokens = synth.zipf_tokens(2_000_000, V, 1.1, seed=77).numpy()
    tokens[::1000] = V + 5  # some invalid
    _count_and_compare(tokens, V)


def test_count_accumulates():
    dev = need_cuda()
    V = 4096
    a = synth.zipf_tokens(300_001, V, 1.1, seed=1).numpy()
    b = synth.zipf_tokens(200_003, V, 1.1, seed=2).numpy()
    counts, n_inv = vt.count_tokens(torch.from_numpy(a).to(dev), V)
    vt.count_tokens(torch.from_numpy(b).to(dev), V, counts=counts,
                    n_invalid=n_inv)
    ref, _ = oracle.count_tokens(np.concatenate([a, b]), V)
    assert np.array_equal(u32_host(counts).astype(np.uint64), ref)


# ----------------------------------------------------------------- select

def _select_and_compare(counts_host: np.ndarray, V_high: int):
    dev = need_cuda()
    counts = torch.from_numpy(counts_host.astype(np.uint32).view(np.int32)).to(
        dev).view(torch.uint32)
    t2f, f2t, sums = vt.select_vocab(counts, V_high)
    ref = oracle.select_vocab(counts_host.astype(np.uint64), V_high)
    assert np.array_equal(t2f.cpu().numpy(), ref["t2f"])
    assert np.array_equal(f2t.cpu().numpy(), ref["f2t"])
    kept, total = (int(x) for x in sums.cpu().tolist())
    assert (kept, total) == (ref["kept"], ref["total"])
    cov = vt.coverage(sums)
    assert cov == ref["coverage"] or (np.isnan(cov) and np.isnan(ref["coverage"]))
    return ref


def test_select_tiny_pipeline():
    cfg = synth.TINY_BUILD
    tokens = synth.zipf_tokens(cfg.n_tokens, cfg.V, cfg.s, cfg.seed).numpy()
    counts, _ = oracle.count_tokens(tokens, cfg.V)
    ref = _select_and_compare(counts, cfg.V_high)
    assert 0.85 < ref["coverage"] < 0.95


@pytest.mark.parametrize("V,V_high,hi,seed", [
    (128256, 32768, 50, 1),          # heavy ties
    (128256, 32768, 2**32 - 1, 2),   # all four digits matter
    (4097, 4097, 1000, 3),           # V_high = V: full sort, ragged tile
    (5000, 1, 3, 4),                 # single kept id, ties at the top
    (1, 1, 10, 5),                   # one-element vocabulary
    (10000, 777, 0, 6),              # all counts zero: ids in order
    (131072, 65536, 300, 7),         # V_high = V / 2, many tiles
    (200000, 32768, 3000, 8),        # V above the Llama-3 vocabulary
])
def test_select_cases(V, V_high, hi, seed):
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, hi, size=V, endpoint=True, dtype=np.uint64)
    _select_and_compare(counts, V_high)


def test_select_zero_total_coverage_nan():
    ref = _select_and_compare(np.zeros(100, np.uint64), 10)
    assert np.isnan(ref["coverage"])


# ----------------------------------------------------------------- gather

def test_gather_ragged_with_invalid_rows():
    dev = need_cuda()
    rng = np.random.default_rng(0)
    V, d, V_high = 5003, 264, 1111
    W = synth.normal_bf16((V, d), 0.02, seed=3).to(dev)
    t2f_h = rng.permutation(V)[:V_high].astype(np.int32)
    t2f_h[5] = -1
    t2f_h[77] = V
    t2f = torch.from_numpy(t2f_h).to(dev)
    n_invalid = torch.zeros(1, dtype=torch.int64, device=dev)
    out = vt.gather_rows(W, t2f, n_invalid=n_invalid)
    ref, rc = oracle.gather_rows(bits_host(W), t2f_h)
    assert rc == 2
    assert np.array_equal(bits_host(out), ref)
    assert int(n_invalid.item()) == 2


def test_gather_full_scale_llama3_8b():
    """128256 x 4096 bf16 weight, the 32768 most frequent rows."""
    dev = need_cuda()
    cfg = synth.SCALE_BUILD
    W = synth.normal_bf16((cfg.V, cfg.d), 0.02, seed=cfg.seed, device=dev)
    t2f = synth.expected_rank_ids(cfg.V, cfg.V_high, cfg.seed).to(dev)
    out = vt.gather_rows(W, t2f)
    ref, rc = oracle.gather_rows(bits_host(W), t2f.cpu().numpy())
    assert rc == 0
    assert np.array_equal(bits_host(out), ref)


# ------------------------------------------------------- full-scale build

def test_vocab_build_full_scale_1e9_tokens():
    """The 1e9-token build of the bench: histogram and selection bit-exact
    against the oracle over the whole stream."""
    dev = need_cuda()
    cfg = synth.SCALE_BUILD
    tokens = synth.zipf_tokens(cfg.n_tokens, cfg.V, cfg.s, cfg.seed, device=dev)
    counts, n_invalid = vt.count_tokens(tokens, cfg.V)
    t2f, f2t, sums = vt.select_vocab(counts, cfg.V_high)
    host_tokens = tokens.cpu().numpy()
    del tokens
    ref_counts, ref_inv = oracle.count_tokens(host_tokens, cfg.V)
    assert np.array_equal(u32_host(counts).astype(np.uint64), ref_counts)
    assert int(n_invalid.item()) == ref_inv == 0
    ref = oracle.select_vocab(ref_counts, cfg.V_high)
    assert np.array_equal(t2f.cpu().numpy(), ref["t2f"])
    assert np.array_equal(f2t.cpu().numpy(), ref["f2t"])
    assert vt.coverage(sums) == ref["coverage"]
    assert 0.93 < ref["coverage"] < 0.95


def test_gather_bias_ragged_with_invalid_ids():
    dev = need_cuda()
    rng = np.random.default_rng(5)
    V, V_high = 70001, 3333
    b = rng.normal(0, 1, V).astype(np.float32)
    t2f_h = rng.permutation(V)[:V_high].astype(np.int32)
    t2f_h[[0, 17, V_high - 1]] = [-5, V, 2**31 - 1]
    n_invalid = torch.zeros(1, dtype=torch.int64, device=dev)
    out = vt.gather_bias(torch.from_numpy(b).to(dev),
                         torch.from_numpy(t2f_h).to(dev), n_invalid=n_invalid)
    ref, bad = oracle.gather_bias(b, t2f_h)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert int(n_invalid.item()) == bad == 3
