"""GPU parity of vt_draft_head_sets (hidden states using different kept
vocabularies) against the CPU oracle run on each hidden state's own set,
through the C ABI: top-k with per-set biases and a temperature, draws whose
noise index is the row in the call, and equality with the plain head when
every row uses one set."""
import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import LOGIT_RTOL, PROB_ATOL, bits_host, check_topk, need_cuda

pytestmark = pytest.mark.gpu


def make_sets(dev, d, V, sizes, seed, bias=True):
    sets = []
    for j, Vh in enumerate(sizes):
        t2f = synth.rank_permutation(V, seed + j)[:Vh].to(dev)
        W = synth.normal_bf16((Vh, d), 0.05, seed=seed + 10 + j, device=dev)
        b = (torch.from_numpy(np.random.default_rng(seed + j).normal(0, 0.4, Vh)
                              .astype(np.float32)).to(dev) if bias else None)
        sets.append((W, t2f, b))
    return sets


@pytest.mark.parametrize("M,k", [(9, 8), (1, 4), (40, 10)])
def test_sets_topk_match_oracle_per_set(M, k):
    dev = need_cuda()
    d, V = 512, 12000
    sets = make_sets(dev, d, V, (3000, 1500, 4096), seed=500 + M)
    H = synth.normal_bf16((M, d), 1.0, seed=600 + M, device=dev)
    sor = np.random.default_rng(M).integers(0, len(sets), M)
    ids, probs = vt.draft_head_sets(H, sor, [s[0] for s in sets],
                                    [s[1] for s in sets], k,
                                    bias_sets=[s[2] for s in sets],
                                    temperature=0.8)
    torch.cuda.synchronize()
    ids, probs = ids.cpu().numpy(), probs.cpu().numpy()
    Hh = bits_host(H)
    for s, (W, t2f, b) in enumerate(sets):
        rows = np.nonzero(sor == s)[0]
        if rows.size == 0:
            continue
        Wh, t2f_h, b_h = bits_host(W), t2f.cpu().numpy(), b.cpu().numpy()
        ref = oracle.draft_head_ex(Hh[rows], Wh, t2f_h, k, bias=b_h,
                                   temperature=0.8)
        lg = (oracle.head_logits(Hh[rows], Wh) + b_h.astype(np.float64)) / 0.8
        # check_topk compares ranks by these scores and probabilities by
        # softmax(scores); the tolerance is scaled for the temperature
        ref_scaled = dict(ref, logits=ref["logits"] / 0.8)
        check_topk(ids[rows], probs[rows], lg, t2f_h, ref_scaled, k)


def test_sets_draws_use_the_row_in_the_call():
    dev = need_cuda()
    d, V, M, k = 256, 9000, 12, 3
    sets = make_sets(dev, d, V, (2000, 3000), seed=700, bias=False)
    H = synth.normal_bf16((M, d), 1.0, seed=701, device=dev)
    sor = np.array([1, 0, 0, 1, 1, 0, 1, 0, 0, 0, 1, 1])
    ids, probs = vt.draft_head_sets(H, sor, [s[0] for s in sets],
                                    [s[1] for s in sets], k, sample=True,
                                    seed=17, offset=3)
    torch.cuda.synchronize()
    ids, probs = ids.cpu().numpy(), probs.cpu().numpy()
    Hh = bits_host(H)
    exact = 0
    for m in range(M):
        W, t2f, _ = sets[sor[m]]
        Wh, t2f_h = bits_host(W), t2f.cpu().numpy()
        ref = oracle.draft_head_ex(Hh[m:m + 1], Wh, t2f_h, k, sample=True,
                                   seed=17, offset=3, m_base=m)
        s_all = oracle.head_logits(Hh[m:m + 1], Wh)[0]
        score = s_all + oracle.gumbel_noise(17, 3, m, t2f_h)
        row_of = {int(f): i for i, f in enumerate(t2f_h)}
        for r in range(k):
            i = row_of[int(ids[m, r])]
            tol = LOGIT_RTOL * (1 + abs(ref["logits"][0, r])) + 1e-4
            assert abs(score[i] - ref["scores"][0, r]) <= tol
            p = np.exp(s_all[i] - ref["row_max"][0]) / ref["row_sumexp"][0]
            assert abs(probs[m, r] - p) <= PROB_ATOL
        exact += int(ids[m].tolist() == ref["ids"][0].tolist())
    assert exact >= M - 1


def test_sets_one_set_equals_plain_head():
    dev = need_cuda()
    d, V, M, k = 1024, 20000, 6, 10
    (W, t2f, _), = make_sets(dev, d, V, (5000,), seed=800, bias=False)
    H = synth.normal_bf16((M, d), 1.0, seed=801, device=dev)
    a = vt.draft_head_sets(H, [0] * M, [W], [t2f], k)
    b = vt.draft_head(H, W, t2f, k)
    assert torch.equal(a[0], b[0])
    torch.testing.assert_close(a[1], b[1], rtol=1e-6, atol=1e-7)
