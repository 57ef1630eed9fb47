"""Seeded random shapes through vt_draft_head against the oracle: d any
multiple of 8, V_high from tens of rows to past the K-split bound, M from
one (GEMV) to 96 (tensor cores, with and without the K split), k from 1 to
32, with and without the remap.  Every logit and the top-k of every row are
checked (run_case in test_gpu_head.py); a second set adds a bias, a
temperature and Gumbel-max draws at random (run_options in
test_gpu_head_options.py), and a third the full-vocabulary q (run_q in
test_gpu_draft_q.py), on both of its paths (the row staged in shared
memory, and past ~57K kept rows the two-launch path).  The shapes are drawn once from a fixed seed, so
a failure names a reproducible case."""
import numpy as np
import pytest

from test_gpu_head import run_case
from test_gpu_head_options import run_options
from test_gpu_draft_q import run_q

pytestmark = pytest.mark.gpu


def _shapes(n=28, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.choice([1, 1, 2, 3, 4, 5, 7, 9, 16, 17, 31, 33, 48, 60, 64, 65, 96]))
        d = int(rng.integers(1, 513)) * 8
        # rows: mostly below the K-split bound (76 tiles of 128), some above
        V_high = int(rng.integers(32, 9728) if i % 4 else rng.integers(9729, 16000))
        # keep the oracle's work (M * V_high * d multiply-adds) modest
        while M * V_high * d > 4e8:
            d = max(8, (d // 2) // 8 * 8)
        k = int(rng.integers(1, min(32, V_high) + 1))
        out.append((d, V_high, M, k, bool(rng.integers(0, 2)), 1000 + i))
    return out


@pytest.mark.parametrize("d,V_high,M,k,use_t2f,seed", _shapes())
def test_random_shape(d, V_high, M, k, use_t2f, seed):
    run_case(d, V_high, M, k, seed=seed, use_t2f=use_t2f)


def _option_shapes(n=16, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i, (d, V_high, M, k, use_t2f, _) in enumerate(_shapes(n, seed)):
        T = float(np.round(rng.uniform(0.5, 1.5), 3))
        out.append((d, V_high, M, k, use_t2f, T, bool(rng.integers(0, 2)),
                    bool(rng.integers(0, 2)), int(rng.integers(0, 2**62)),
                    int(rng.integers(0, 2**40)), 2000 + i))
    return out


@pytest.mark.parametrize("d,V_high,M,k,use_t2f,T,use_bias,sample,gen_seed,offset,seed",
                         _option_shapes())
def test_random_options(d, V_high, M, k, use_t2f, T, use_bias, sample, gen_seed,
                        offset, seed):
    run_options(d, V_high, M, k, seed, T=T, use_bias=use_bias, sample=sample,
                gen_seed=gen_seed, offset=offset, use_t2f=use_t2f)


def _q_shapes(n=12, seed=20261204):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        V_high = int(rng.integers(1, 12000) if i % 3 else rng.integers(57000, 70000))
        V = V_high + int(rng.integers(0, 3 * V_high + 1))
        M = int(rng.choice([1, 2, 3, 5, 8, 13, 21]))
        d = int(rng.integers(1, 129)) * 8
        while M * V_high * d > 3e8:
            d = max(8, (d // 2) // 8 * 8)
        out.append((d, V, V_high, M, float(np.round(rng.uniform(0.5, 1.5), 3)),
                    bool(rng.integers(0, 2)), 3000 + i))
    return out


@pytest.mark.parametrize("d,V,V_high,M,T,use_bias,seed", _q_shapes())
def test_random_q(d, V, V_high, M, T, use_bias, seed):
    run_q(d, V, V_high, M, seed, T=T, use_bias=use_bias)
