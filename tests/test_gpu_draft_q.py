"""GPU parity of the full-vocabulary draft distribution (vt_draft_q) against
the CPU oracle through the C ABI: the GPU head's logits (bias included) turned
into q[M, V] by the library, compared element by element with the oracle's q
computed from the same H and W (within 1e-4, exactly 0 at dropped ids, rows
summing to 1), on ragged and full sizes, with and without the identity map."""
import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import PROB_ATOL, bits_host, need_cuda, oracle_q

pytestmark = pytest.mark.gpu


def f2t_of(t2f_h: np.ndarray, V: int) -> np.ndarray:
    f2t = np.full(V, -1, dtype=np.int32)
    f2t[t2f_h] = np.arange(t2f_h.size, dtype=np.int32)
    return f2t


def run_q(d, V, V_high, M, seed, T=1.0, use_bias=False, identity=False):
    """Every row of q against the oracle."""
    dev = need_cuda()
    W = synth.normal_bf16((V_high, d), 0.02, seed=seed, device=dev)
    H = synth.normal_bf16((M, d), 1.0, seed=seed + 1, device=dev)
    if identity:
        assert V == V_high
        t2f_h, t2f, f2t = None, None, None
    else:
        t2f_h = synth.rank_permutation(V, seed)[:V_high].numpy()
        t2f = torch.from_numpy(t2f_h).to(dev)
        f2t = torch.from_numpy(f2t_of(t2f_h, V)).to(dev)
    b_h = (np.random.default_rng(seed).normal(0, 0.5, V_high).astype(np.float32)
           if use_bias else None)
    bias = None if b_h is None else torch.from_numpy(b_h).to(dev)
    logits = torch.empty(M, V_high, dtype=torch.float32, device=dev)
    vt.draft_head(H, W, t2f, 1, out_logits=logits, bias=bias, temperature=T)
    q = vt.draft_q(logits, f2t, V, temperature=T)
    torch.cuda.synchronize()
    ref = oracle_q(bits_host(H), bits_host(W), t2f_h, V, bias=b_h,
                   temperature=T)
    got = q.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= PROB_ATOL
    if t2f_h is not None:
        dropped = np.setdiff1d(np.arange(V), t2f_h)
        assert np.all(got[:, dropped] == 0.0)
    np.testing.assert_allclose(got.sum(axis=1), 1.0, atol=1e-4)
    return q, logits


@pytest.mark.parametrize("d,V,V_high,M,T,bias", [
    (264, 5003, 1111, 3, 0.8, True),     # ragged V: scalar path
    (512, 4096, 4096, 2, 1.0, False),    # V_high = V with a permuted map
    (256, 9000, 1, 1, 1.0, False),       # one kept id: q is one-hot
    (1032, 20000, 3001, 7, 1.7, True),   # vector path, several rows
])
def test_q_shapes(d, V, V_high, M, T, bias):
    q, _ = run_q(d, V, V_high, M, seed=V + M, T=T, use_bias=bias)
    if V_high == 1:
        assert float(q.max()) == 1.0


def test_q_identity_map():
    run_q(1024, 3000, 3000, 2, seed=5, T=0.7, identity=True)


def test_q_full_size_llama3_8b():
    """The 8B shape: 32768 kept of 128256, one hidden state."""
    run_q(4096, 128256, 32768, 1, seed=1002)


def test_q_tree_m60_every_row():
    """The EAGLE-2 tree step: q of all 60 nodes over V = 128256."""
    run_q(4096, 128256, 32768, 60, seed=1003, T=0.9)


def test_q_at_drawn_tokens_is_the_reported_probability():
    """The probability the sampling head reports for its draw is q there."""
    dev = need_cuda()
    V, V_high, d, M = 12000, 3000, 512, 5
    W = synth.normal_bf16((V_high, d), 0.05, seed=71, device=dev)
    H = synth.normal_bf16((M, d), 1.0, seed=72, device=dev)
    t2f_h = synth.rank_permutation(V, 73)[:V_high].numpy()
    t2f = torch.from_numpy(t2f_h).to(dev)
    f2t = torch.from_numpy(f2t_of(t2f_h, V)).to(dev)
    logits = torch.empty(M, V_high, dtype=torch.float32, device=dev)
    for Mx in (1, M):
        ids, probs = vt.draft_head(H[:Mx], W, t2f, 3, out_logits=logits[:Mx],
                                   sample=True, seed=4, offset=9,
                                   temperature=0.6)
        q = vt.draft_q(logits[:Mx], f2t, V, temperature=0.6)
        torch.testing.assert_close(torch.gather(q, 1, ids.long()), probs,
                                   rtol=1e-5, atol=1e-7)
