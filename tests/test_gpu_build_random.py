"""Seeded random cases of the offline build against the oracle, bit-exact:
token streams of random length, vocabulary, Zipf exponent and share of
invalid ids through vt_count_tokens, the resulting counts (and random
counts with many ties) through vt_select_vocab, and random row maps through
vt_gather_rows.  The cases are drawn once from a fixed seed."""
import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import bits_host, need_cuda
from test_gpu_build import _count_and_compare, _select_and_compare

pytestmark = pytest.mark.gpu


def _build_cases(n=16, seed=20261205):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        V = int(rng.choice([7, 300, 4096, 4097, 32000, 128256, 151936, 250001]))
        n_tok = int(rng.integers(0, 3_000_000))
        s = float(np.round(rng.uniform(0.6, 1.6), 2))
        bad = float(rng.choice([0.0, 0.0, 0.01, 0.3]))
        V_high = int(rng.integers(1, V + 1))
        out.append((V, n_tok, s, bad, V_high, 4000 + i))
    return out


@pytest.mark.parametrize("V,n_tok,s,bad,V_high,seed", _build_cases())
def test_random_count_then_select(V, n_tok, s, bad, V_high, seed):
    rng = np.random.default_rng(seed)
    tokens = synth.zipf_tokens(n_tok, V, s, seed=seed).numpy().copy()
    if bad and n_tok:
        hit = rng.random(n_tok) < bad
        tokens[hit] = rng.choice([-1, V, V + 7, 2**31 - 1, -(2**31)], hit.sum())
    got = _count_and_compare(tokens, V)
    _select_and_compare(got.astype(np.uint64), V_high)


@pytest.mark.parametrize("seed", range(6))
def test_random_select_with_ties(seed):
    rng = np.random.default_rng(5000 + seed)
    V = int(rng.integers(1, 200_000))
    hi = int(rng.choice([0, 1, 7, 255, 256, 65535, 2**24, 2**32 - 1]))
    counts = rng.integers(0, hi, size=V, endpoint=True, dtype=np.uint64)
    _select_and_compare(counts, int(rng.integers(1, V + 1)))


@pytest.mark.parametrize("seed", range(6))
def test_random_gather(seed):
    dev = need_cuda()
    rng = np.random.default_rng(6000 + seed)
    V = int(rng.integers(1, 20000))
    d = int(rng.integers(1, 513)) * 8
    V_high = int(rng.integers(1, V + 1))
    W = synth.normal_bf16((V, d), 0.02, seed=6000 + seed, device=dev)
    t2f = rng.permutation(V)[:V_high].astype(np.int32)
    got = vt.gather_rows(W, torch.from_numpy(t2f).to(dev))
    ref, rc = oracle.gather_rows(bits_host(W), t2f)
    assert rc == 0
    assert np.array_equal(bits_host(got), ref)
