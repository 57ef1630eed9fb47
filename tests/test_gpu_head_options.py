"""GPU parity of the head's options (vt_draft_head_ex) against the CPU
oracle, through the C ABI: the sampler's noise value by value, bias and
temperature on both head paths, Gumbel-max draws (k = 1) and draws without
replacement (k > 1) id by id, the law of the drawn ids, and the invariance
of draws under trimming."""
import numpy as np
import pytest
import torch
from scipy import stats

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import (LOGIT_RTOL, PROB_ATOL, bits_host, check_logits,
                      need_cuda, oracle_head)

pytestmark = pytest.mark.gpu

NOISE_TOL = 1e-4  # fp32 logs of an exact uniform: actual error ~1e-6


def check_selection(ids, probs, logits, s, score, t2f_h, ref, k, T):
    """Rank r of the GPU's answer names a kept row whose oracle score is
    within tolerance of the oracle's r-th score (ids differ from the
    oracle's only at near-ties), ids are distinct, and each probability is
    the oracle's softmax(logit / T) of that id.  Returns the exact rows."""
    M, V_high = s.shape
    row_of = ({int(f): i for i, f in enumerate(t2f_h)} if t2f_h is not None
              else None)
    exact = 0
    for m in range(M):
        g = ids[m].tolist()
        assert len(set(g)) == k, f"row {m}: repeated ids {g}"
        for r in range(k):
            gid = int(g[r])
            row = gid if row_of is None else row_of.get(gid)
            assert row is not None and 0 <= row < V_high, f"row {m}: id {gid} not kept"
            tol = LOGIT_RTOL * (1 + abs(ref["logits"][m, r])) / T + NOISE_TOL
            assert abs(score[m, row] - ref["scores"][m, r]) <= tol, (
                f"row {m} rank {r}: gpu id {gid} score {score[m, row]} vs "
                f"oracle id {ref['ids'][m, r]} score {ref['scores'][m, r]}")
            p_ref = np.exp(s[m, row] - ref["row_max"][m]) / ref["row_sumexp"][m]
            assert abs(float(probs[m, r]) - p_ref) <= PROB_ATOL, (
                f"row {m} rank {r}: prob {probs[m, r]} vs {p_ref}")
        exact += int(g == ref["ids"][m].tolist())
    return exact


def run_options(d, V_high, M, k, seed, T=1.0, use_bias=False, sample=False,
                gen_seed=0, offset=0, use_t2f=True):
    """Every hidden state of the call against the oracle."""
    dev = need_cuda()
    W = synth.normal_bf16((V_high, d), 0.02, seed=seed, device=dev)
    H = synth.normal_bf16((M, d), 1.0, seed=seed + 1, device=dev)
    t2f = synth.rank_permutation(2 * V_high, seed)[:V_high].to(dev) if use_t2f else None
    bias = (torch.from_numpy(np.random.default_rng(seed).normal(0, 0.5, V_high)
                             .astype(np.float32)).to(dev) if use_bias else None)
    logits = torch.empty(M, V_high, dtype=torch.float32, device=dev)
    ws = torch.zeros(vt.workspace_bytes("head", M=M, k=k, V_high=V_high),
                     dtype=torch.uint8, device=dev)
    ids, probs = vt.draft_head(H, W, t2f, k, out_logits=logits, ws=ws, bias=bias,
                               temperature=T, sample=sample, seed=gen_seed,
                               offset=offset)
    torch.cuda.synchronize()
    assert int(ws[128:132].view(torch.int32).item()) == 0, "device error word"
    Hh, Wh = bits_host(H), bits_host(W)
    t2f_h = None if t2f is None else t2f.cpu().numpy()
    b_h = None if bias is None else bias.cpu().numpy()
    ref, lg = oracle_head(Hh, Wh, t2f_h, k, bias=b_h, temperature=T,
                          sample=sample, seed=gen_seed, offset=offset)
    if b_h is not None:
        lg = lg + b_h.astype(np.float64)[None, :]
    s = lg / T
    score = s.copy()
    if sample:  # the noise is keyed by the hidden state's row in the call
        fids = np.arange(V_high, dtype=np.int32) if t2f_h is None else t2f_h
        for m in range(M):
            score[m] += oracle.gumbel_noise(gen_seed, offset, m, fids)
    check_logits(logits.cpu().numpy(), lg)
    return check_selection(ids.cpu().numpy(), probs.cpu().numpy(), lg, s,
                           score, t2f_h, ref, k, T)


def test_noise_matches_oracle():
    """The device generator against the oracle's: the uniform is exact on
    both sides, so the noise differs only by fp32 rounding of the logs."""
    dev = need_cuda()
    ids = np.concatenate([np.arange(0, 5000), [2**31 - 1, 2**31 - 2, 128255],
                          np.random.default_rng(1).integers(0, 2**31 - 1, 5000)]
                         ).astype(np.int32)
    ids_d = torch.from_numpy(ids).to(dev)
    for seed, offset, m in [(0, 0, 0), (12345, 7, 3), (2**63 + 5, 2**40 + 9, 255),
                            (2**32, 2**32 - 1, 1)]:
        g = vt.draft_noise(seed, offset, m, ids_d).cpu().numpy().astype(np.float64)
        ref = oracle.gumbel_noise(seed, offset, m, ids)
        np.testing.assert_allclose(g, ref, rtol=2e-6, atol=2e-6)


@pytest.mark.parametrize("M", [1, 3, 40])
def test_topk_with_bias_and_temperature(M):
    exact = run_options(1032, 3001, M, 10, seed=200 + M, T=0.7, use_bias=True)
    assert exact >= M - 1


@pytest.mark.parametrize("M,k,T,use_bias", [(1, 1, 1.0, False), (1, 8, 0.6, True),
                                            (2, 1, 1.0, True), (4, 5, 1.5, False),
                                            (60, 1, 0.8, False), (33, 10, 1.0, True)])
def test_sampled_ids_match_oracle(M, k, T, use_bias):
    """Gumbel-max draws (k = 1) and draws without replacement (k > 1):
    the GPU draws the oracle's ids except at score near-ties."""
    for offset in (0, 1, 2**33 + 3):
        exact = run_options(520, 2000, M, k, seed=300 + M + k, T=T,
                            use_bias=use_bias, sample=True, gen_seed=77 + M,
                            offset=offset)
        assert exact >= M - 1


def test_sampled_full_size_llama3_8b():
    """The Llama-3-8B-shaped draft step, sampling at temperature 0.8."""
    for offset in (5, 6):
        run_options(4096, 32768, 1, 1, seed=1002, T=0.8, sample=True,
                    gen_seed=2026, offset=offset)


def test_sampled_tree_m60_every_row():
    """The EAGLE-2 tree step (M = 60) drawing four tokens per node: every
    node against the oracle."""
    exact = run_options(4096, 32768, 60, 4, seed=1003, sample=True, gen_seed=9,
                        offset=1)
    assert exact >= 58


@pytest.mark.parametrize("M", [1, 120])
def test_draw_law_on_gpu(M):
    """Logits exact by construction (one-hot hidden states against chosen
    values): 6000 draws over offsets (and hidden states) follow
    softmax((l + b) / T) (chi-square)."""
    dev = need_cuda()
    values = np.array([0.5, 1.0, -0.25, 2.0, 0.0, 1.5, -1.0, 0.75, 0.25, -0.5,
                       1.25, 0.125, -2.0, 0.375, 1.75, -0.125], np.float32)
    bias = np.linspace(-0.3, 0.3, values.size).astype(np.float32)
    T = 0.7
    d = 64
    W = np.zeros((values.size, d), np.float32)
    W[:, 0] = values
    Hn = np.zeros((M, d), np.float32)
    Hn[:, 0] = 1.0
    Wd = torch.from_numpy(W).to(torch.bfloat16).to(dev)
    Hd = torch.from_numpy(Hn).to(torch.bfloat16).to(dev)
    bd = torch.from_numpy(bias).to(dev)
    draws = []
    for offset in range(6000 // M):
        ids, _ = vt.draft_head(Hd, Wd, None, 1, bias=bd, temperature=T,
                               sample=True, seed=31337, offset=offset)
        draws.append(ids[:, 0])
    counts = np.bincount(torch.cat(draws).cpu().numpy(), minlength=values.size)
    lb = (values.astype(np.float64) + bias) / T
    p = np.exp(lb - lb.max())
    p /= p.sum()
    assert stats.chisquare(counts, counts.sum() * p).pvalue > 1e-4


def test_trimmed_draw_equals_untrimmed_draw_when_kept():
    """Same seed and step: the trimmed head draws the untrimmed head's token
    whenever that token is kept (noise is keyed by full id)."""
    dev = need_cuda()
    V, d, M = 8192, 256, 200
    Wf = synth.normal_bf16((V, d), 0.2, seed=51, device=dev)
    H = synth.normal_bf16((M, d), 1.0, seed=52, device=dev)
    t2f = synth.rank_permutation(V, 53)[:2048].to(dev)
    W_high = vt.gather_rows(Wf, t2f)
    for Mx in (1, M):
        full, _ = vt.draft_head(H[:Mx], Wf, None, 1, sample=True, seed=8,
                                offset=21, temperature=0.5)
        trim, _ = vt.draft_head(H[:Mx], W_high, t2f, 1, sample=True, seed=8,
                                offset=21, temperature=0.5)
        f, t = full[:, 0].cpu().numpy(), trim[:, 0].cpu().numpy()
        kept = np.isin(f, t2f.cpu().numpy())
        assert np.array_equal(f[kept], t[kept])
        if Mx == M:
            assert kept.sum() >= 25  # about a quarter of 200 expected


def test_topk_options_default_equal_plain_call():
    """vt_draft_head_ex with default options is vt_draft_head."""
    dev = need_cuda()
    W = synth.normal_bf16((5000, 1024), 0.02, seed=61, device=dev)
    for M in (1, 6):
        H = synth.normal_bf16((M, 1024), 1.0, seed=62, device=dev)
        a = vt.draft_head(H, W, None, 10)
        a = [t.clone() for t in a]
        b = vt.draft_head(H, W, None, 10, temperature=1.0, bias=torch.zeros(
            5000, dtype=torch.float32, device=dev))
        assert torch.equal(a[0], b[0])
        torch.testing.assert_close(a[1], b[1], rtol=1e-6, atol=1e-7)
