"""The README's Python example, at small sizes: build the kept vocabulary
from a token stream and a head, save it, and draft with it (top-k, a draw
and the full-vocabulary q), each result checked against the oracle or a
plain definition."""
import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import bits_host, check_topk, need_cuda

pytestmark = pytest.mark.gpu


def test_readme_example(tmp_path):
    dev = need_cuda()
    V, V_high, d, M, k = 4096, 1024, 256, 3, 10
    tokens = synth.zipf_tokens(200_000, V, 1.1, seed=71).to(dev)
    lm_head = synth.normal_bf16((V, d), 0.02, seed=72, device=dev)
    h = synth.normal_bf16((M, d), 1.0, seed=73, device=dev)

    vocab = vt.build_vocab(tokens, V=V, V_high=V_high, W=lm_head)
    counts, _ = oracle.count_tokens(tokens.cpu().numpy(), V)
    sel = oracle.select_vocab(counts, V_high)
    assert vocab["t2f"].cpu().numpy().tolist() == sel["t2f"].tolist()
    assert vt.coverage(vocab["sums"]) == sel["coverage"]
    vt.save_vocab(str(tmp_path / "vocab.npz"), vocab)
    again = vt.load_vocab(str(tmp_path / "vocab.npz"), device=dev)
    assert torch.equal(again["t2f"], vocab["t2f"])

    logits = torch.empty(M, V_high, dtype=torch.float32, device=dev)
    ids, probs = vt.draft_head(h, vocab["W_high"], vocab["t2f"], k=k,
                               out_logits=logits)
    Hh, Wh, t2f_h = bits_host(h), bits_host(vocab["W_high"]), sel["t2f"]
    ref = oracle.draft_head(Hh, Wh, t2f_h, k)
    check_topk(ids.cpu().numpy(), probs.cpu().numpy(), oracle.head_logits(Hh, Wh),
               t2f_h, ref, k)

    drawn, p1 = vt.draft_head(h, vocab["W_high"], vocab["t2f"], k=1,
                              sample=True, seed=1234, offset=5)
    assert set(drawn.cpu().numpy().ravel().tolist()) <= set(t2f_h.tolist())
    assert bool((p1 > 0).all())

    q = vt.draft_q(logits, vocab["f2t"], V)
    assert q.shape == (M, V)
    kept = torch.zeros(V, dtype=torch.bool, device=dev)
    kept[vocab["t2f"].long()] = True
    assert bool((q[:, ~kept] == 0).all())
    torch.testing.assert_close(q.sum(dim=1), torch.ones(M, device=dev), rtol=0, atol=1e-5)
    # q at each top-k id is the probability the head reported for it
    torch.testing.assert_close(q.gather(1, ids.long()), probs, rtol=1e-4, atol=1e-6)
