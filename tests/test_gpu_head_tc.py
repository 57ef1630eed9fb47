"""GPU parity of the tree-draft (tensor-core) head path, M >= 2 hidden
states, against the CPU oracle through the C ABI: logits within
1e-3 * (1 + |l|), probabilities within 1e-4, top-k ids equal to the
oracle's except where oracle logits are closer than that tolerance.  Sizes
cover ragged K blocks (d not a multiple of 64), ragged last tiles (V_high
not a multiple of 128), N = M rounded up to 16 from 16 to 256, and the
full EAGLE-2 tree-draft shapes (sampled hidden states)."""
import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import (bits_host, check_logits, check_topk, fp32_sum_bound,
                      need_cuda, oracle_head)

pytestmark = pytest.mark.gpu


def run_tc(d, V_high, M, k, seed, use_t2f=True, want_logits=True,
           hs=1.0, ws_scale=0.02, widen=False):
    """Every hidden state of the call against the oracle."""
    dev = need_cuda()
    W_high = synth.normal_bf16((V_high, d), ws_scale, seed=seed, device=dev)
    H = synth.normal_bf16((M, d), hs, seed=seed + 1, device=dev)
    t2f = (synth.rank_permutation(2 * V_high, seed)[:V_high].to(dev)
           if use_t2f else None)
    ws = torch.zeros(vt.workspace_bytes("head", M=M, k=k, V_high=V_high),
                     dtype=torch.uint8, device=dev)
    logits = (torch.empty(M, V_high, dtype=torch.float32, device=dev)
              if want_logits else None)
    ids, probs = vt.draft_head(H, W_high, t2f, k, out_logits=logits, ws=ws)
    torch.cuda.synchronize()
    err = int(ws[128:132].view(torch.int32).item())
    assert err == 0, f"device error word {err}"
    Hh, Wh = bits_host(H), bits_host(W_high)
    t2f_h = None if t2f is None else t2f.cpu().numpy()
    ref, ref_logits = oracle_head(Hh, Wh, t2f_h, k)
    extra = fp32_sum_bound(Hh, Wh) if widen else None
    if want_logits:
        check_logits(logits.cpu().numpy(), ref_logits,
                     0.0 if extra is None else extra)
    check_topk(ids.cpu().numpy(), probs.cpu().numpy(), ref_logits, t2f_h, ref,
               k, extra)
    return ids, probs


@pytest.mark.parametrize("d,V_high,M,k", [
    (256, 1024, 2, 8),       # smallest M on this path: N = 16
    (256, 1024, 5, 8),
    (1032, 3001, 16, 10),    # ragged K block and ragged last tile
    (2048, 4096, 33, 10),    # N = 48
    (520, 777, 64, 1),       # greedy, one partial tile only
    (3584, 2000, 128, 32),   # N = 128, k = 32
    (512, 1500, 256, 5),     # N = 256, the widest MMA
])
def test_tc_shapes(d, V_high, M, k):
    run_tc(d, V_high, M, k, seed=d + V_high + M)


@pytest.mark.parametrize("d,V_high,M,k", [
    (520, 1000, 9, 10),      # 9 K atoms, 3 stages: halves of 1 and 2 stages
    (1000, 4000, 20, 7),     # ragged last K atom (1000 = 15 x 64 + 40)
    (4096, 9728, 60, 10),    # 76 tiles on 152 SMs: the largest split grid
    (2056, 257, 64, 32),     # one full tile and one row, N = 64
    (8200, 640, 3, 4),       # long K, N = 16
    (1024, 3000, 200, 10),   # N = 208: several 16-column chunks per epilogue warp
    (512, 2000, 256, 5),     # N = 256: the widest exchange buffer
])
def test_tc_k_split_between_cluster_pairs(d, V_high, M, k):
    """With at most half as many 128-row tiles as SMs (and at least eight K
    atoms), the two CTAs of a cluster each sum half of a tile's K stages and
    exchange partial sums through distributed shared memory; every logit and
    the top-k against the oracle, odd stage counts and ragged K included."""
    run_tc(d, V_high, M, k, seed=d + V_high + M)


def test_tc_identity_map():
    run_tc(1024, 5000, 24, 10, seed=3, use_t2f=False)


def test_tc_large_logits_no_overflow():
    """Huge, cancelling products: logits are held to the fp32 summation
    bound on top of the usual tolerance; the softmax must not overflow."""
    _, probs = run_tc(1024, 3000, 8, 10, seed=4, hs=64.0, ws_scale=1.0,
                      widen=True)
    assert torch.isfinite(probs).all()


def test_tc_repeated_calls_identical():
    dev = need_cuda()
    W = synth.normal_bf16((10000, 2048), 0.02, seed=7, device=dev)
    H = synth.normal_bf16((20, 2048), 1.0, seed=8, device=dev)
    a = [t.clone() for t in vt.draft_head(H, W, None, 10)]
    for _ in range(3):
        ids, probs = vt.draft_head(H, W, None, 10)
        assert torch.equal(ids, a[0]) and torch.equal(probs, a[1])


@pytest.mark.parametrize("V_high", [8192, 16384, 32768, 65536])
def test_tc_eagle2_tree_m60_v_high_sweep(V_high):
    """EAGLE-2-style tree draft, d = 4096, M = 60, over the V_high sweep
    (8192 .. 65536): every hidden state against the oracle, logits
    included."""
    run_tc(4096, V_high, 60, 10, seed=1003 + V_high)


def test_tc_full_vocab_m60_every_row():
    """The untrimmed end of the sweep (V = 128256, identity map), every
    hidden state against the oracle."""
    run_tc(4096, 128256, 60, 10, seed=1003, use_t2f=False)


@pytest.mark.parametrize("shape", [synth.QWEN7B_HEAD, synth.LLAMA1B_HEAD])
@pytest.mark.parametrize("M", [16, 64])
def test_tc_qwen_and_llama1b_batch_sweep(shape, M):
    run_tc(shape.d, shape.V_high, M, shape.k, seed=shape.seed + M)


def test_gemv_and_tc_paths_share_one_workspace():
    """One workspace serves calls of any M: the small-M and tree-draft paths
    keep their counters in separate parts of the shared header, so
    alternating them (the order that once left stale counters) stays exact."""
    dev = need_cuda()
    V_high, d, k = 6000, 1024, 10
    W = synth.normal_bf16((V_high, d), 0.02, seed=41, device=dev)
    Hs = {M: synth.normal_bf16((M, d), 1.0, seed=42 + M, device=dev)
          for M in (1, 9, 3, 40)}
    nbytes = max(vt.workspace_bytes("head", M=M, k=k, V_high=V_high) for M in Hs)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    Wh = bits_host(W)
    for M in (1, 9, 3, 40, 1, 9):
        ids, probs = vt.draft_head(Hs[M], W, None, k, ws=ws)
        torch.cuda.synchronize()
        Hh = bits_host(Hs[M])
        ref = oracle.draft_head(Hh, Wh, None, k)
        check_topk(ids.cpu().numpy(), probs.cpu().numpy(),
                   oracle.head_logits(Hh, Wh), None, ref, k)


def test_tc_row_survivor_worst_case_k32():
    """k = 32 with one low-scoring thread in every warp of a row part: the
    part's bound T is then low and nearly every value of the 4096-value part
    survives it; all of them must be ranked (none dropped), so the ids equal
    the oracle's exactly (logits exact: one-hot hidden states)."""
    dev = need_cuda()
    V_high, d, M, k = 8192, 64, 3, 32
    rng = np.random.default_rng(90)
    vals = 1.0 + rng.integers(0, 128, V_high) / 128.0  # bf16-exact
    i = np.arange(V_high)
    t = ((i % 4096) % 1024) // 4  # thread of the part holding index i
    vals[t % 32 == 0] = -5.0
    W = np.zeros((V_high, d), np.float32)
    W[:, 0] = vals
    Hn = np.zeros((M, d), np.float32)
    Hn[:, 0] = 1.0
    Wd = torch.from_numpy(W).to(torch.bfloat16).to(dev)
    Hd = torch.from_numpy(Hn).to(torch.bfloat16).to(dev)
    t2f = synth.rank_permutation(2 * V_high, 91)[:V_high].to(dev)
    ids, probs = vt.draft_head(Hd, Wd, t2f, k)
    torch.cuda.synchronize()
    ref = oracle.draft_head(bits_host(Hd), bits_host(Wd), t2f.cpu().numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    np.testing.assert_allclose(probs.cpu().numpy(), ref["probs"], atol=1e-6)


@pytest.mark.parametrize("V_high", [32768, 32771])
def test_tc_all_quadrants_reach_the_bound(V_high):
    """Every 32-row quadrant holds one logit of exactly 2.0 and the rest
    below: the bound on the k-th best score equals 2.0, every quadrant
    reaches it (more than can be read one by one), so the row is scanned
    whole; the 2.0 entries tie and the k with the lowest full ids win, as in
    the oracle (logits exact: one-hot hidden states)."""
    dev = need_cuda()
    d, M, k = 64, 2, 10
    rng = np.random.default_rng(V_high)
    vals = 1.0 + rng.integers(0, 64, V_high) / 128.0  # bf16-exact, < 2
    top = np.arange(0, V_high, 32) + rng.integers(0, 32, (V_high + 31) // 32)
    vals[top[top < V_high]] = 2.0
    W = np.zeros((V_high, d), np.float32)
    W[:, 0] = vals
    Hn = np.zeros((M, d), np.float32)
    Hn[:, 0] = 1.0
    Wd = torch.from_numpy(W).to(torch.bfloat16).to(dev)
    Hd = torch.from_numpy(Hn).to(torch.bfloat16).to(dev)
    t2f = synth.rank_permutation(2 * V_high, 92)[:V_high].to(dev)
    ids, probs = vt.draft_head(Hd, Wd, t2f, k)
    torch.cuda.synchronize()
    ref = oracle.draft_head(bits_host(Hd), bits_host(Wd), t2f.cpu().numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    np.testing.assert_allclose(probs.cpu().numpy(), ref["probs"], atol=1e-6)
