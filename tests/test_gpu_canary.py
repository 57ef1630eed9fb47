"""Guard bands around every device output, on the GPU.

Each output (and each workspace) is the middle of a larger buffer whose
4 KiB on either side hold a known byte pattern; after the call the pattern
must be intact byte for byte, so no kernel writes before the start or past
the end of what the call owns.  Shapes are ragged on purpose (V_high not a
multiple of the 128-row tile, d not a multiple of 64, V % 4 != 0, k not a
power of two), where vectorised tails and partial tiles are written.  A
light check of each result against the oracle or a library routine shows
the call did write its output.  (Sanitizer tools are not available on
these GPUs; this is the bounds evidence.)"""
import ctypes

import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import bits_host, check_topk, need_cuda, oracle_head

pytestmark = pytest.mark.gpu

PAD = 4096
PATTERN = 0xA5


class Guarded:
    """A tensor of ``shape`` and ``dtype`` with PAD pattern bytes on both
    sides (the tensor starts 4096 bytes into a fresh allocation, so it keeps
    the allocation's alignment)."""

    def __init__(self, shape, dtype, dev, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.buf = torch.full((PAD + n + PAD,), PATTERN, dtype=torch.uint8,
                              device=dev)
        self.t = self.buf[PAD:PAD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, name):
        torch.cuda.synchronize()
        head = self.buf[:PAD].cpu().numpy()
        tail = self.buf[PAD + self.n:].cpu().numpy()
        bad_h = np.nonzero(head != PATTERN)[0]
        bad_t = np.nonzero(tail != PATTERN)[0]
        assert bad_h.size == 0, f"{name}: {bad_h.size} bytes written before the start (first at -{PAD - bad_h[0]})"
        assert bad_t.size == 0, f"{name}: {bad_t.size} bytes written past the end (first at +{bad_t[0]})"


def ws_for(op, dev, **kw):
    return Guarded((vt.workspace_bytes(op, **kw),), torch.uint8, dev, fill=0)


@pytest.mark.parametrize("n,V", [(100_003, 5003), (1_000_000, 4096),
                                 (777, 300_001)])
def test_count_tokens_bounds(n, V):
    dev = need_cuda()
    tok = synth.zipf_tokens(n, V, 1.1, seed=V).numpy().copy()
    tok[::97] = -3          # invalid ids
    tok[1::89] = V
    counts = Guarded((V,), torch.int32, dev, fill=0)
    n_inv = Guarded((1,), torch.int64, dev, fill=0)
    ws = ws_for("count", dev, V=V)
    vt.count_tokens(torch.from_numpy(tok).to(dev), V,
                    counts=counts.t.view(torch.uint32), n_invalid=n_inv.t,
                    ws=ws.t)
    for g, name in ((counts, "counts"), (n_inv, "n_invalid"), (ws, "ws")):
        g.check(name)
    valid = tok[(tok >= 0) & (tok < V)]
    assert np.array_equal(counts.t.cpu().numpy(), np.bincount(valid, minlength=V))
    assert int(n_inv.t.item()) == n - valid.size


@pytest.mark.parametrize("V,V_high", [(5003, 1111), (4096, 4096), (300_001, 1)])
def test_select_vocab_bounds(V, V_high):
    dev = need_cuda()
    c = np.random.default_rng(V).integers(0, 50, V).astype(np.uint32)
    counts = torch.from_numpy(c.view(np.int32)).to(dev).view(torch.uint32)
    t2f = Guarded((V_high,), torch.int32, dev)
    f2t = Guarded((V,), torch.int32, dev)
    sums = Guarded((2,), torch.int64, dev)
    ws = Guarded((vt.workspace_bytes("select", V=V),), torch.uint8, dev)
    vt.select_vocab(counts, V_high, ws=ws.t, out=(t2f.t, f2t.t, sums.t))
    for g, name in ((t2f, "t2f"), (f2t, "f2t"), (sums, "sums"), (ws, "ws")):
        g.check(name)
    order = np.lexsort((np.arange(V), -c.astype(np.int64)))
    assert np.array_equal(t2f.t.cpu().numpy(), order[:V_high])


@pytest.mark.parametrize("V,d,V_high", [(5003, 1032, 3001), (4096, 8, 1),
                                        (9000, 264, 777)])
def test_gather_bounds(V, d, V_high):
    dev = need_cuda()
    W = synth.normal_bf16((V, d), 0.02, seed=V, device=dev)
    t2f_h = synth.rank_permutation(V, V + 1)[:V_high].numpy().copy()
    t2f_h[0] = V + 5  # an invalid row: written as zeros, counted
    t2f = torch.from_numpy(t2f_h).to(dev)
    out = Guarded((V_high, d), torch.bfloat16, dev)
    n_inv = Guarded((1,), torch.int64, dev, fill=0)
    vt.gather_rows(W, t2f, out=out.t, n_invalid=n_inv.t)
    out.check("W_high")
    n_inv.check("n_invalid")
    got = bits_host(out.t)
    assert np.array_equal(got[1:], bits_host(W)[t2f_h[1:]])
    assert not got[0].any() and int(n_inv.t.item()) == 1
    b = torch.from_numpy(np.random.default_rng(V).normal(0, 1, V)
                         .astype(np.float32)).to(dev)
    bh = Guarded((V_high,), torch.float32, dev)
    n_inv2 = Guarded((1,), torch.int64, dev, fill=0)
    vt.gather_bias(b, t2f, out=bh.t, n_invalid=n_inv2.t)
    bh.check("b_high")
    n_inv2.check("n_invalid (bias)")
    ref, bad = oracle.gather_bias(b.cpu().numpy(), t2f_h)
    assert np.array_equal(bh.t.cpu().numpy(), ref) and bad == 1


@pytest.mark.parametrize("d,V_high,M,k,sample", [
    (1032, 3001, 1, 10, False),   # GEMV, ragged
    (1032, 3001, 3, 7, True),     # GEMV, several rows, drawing
    (264, 777, 1, 32, False),
    (1032, 3001, 2, 10, False),   # tensor cores, smallest M, ragged tile
    (520, 4099, 17, 5, False),    # N = 32, ragged K and tile
    (1032, 3001, 60, 10, True),   # tensor cores, drawing (per-part rows)
    (264, 130, 100, 32, False),   # one partial tile, k = 32
])
def test_draft_head_bounds(d, V_high, M, k, sample):
    dev = need_cuda()
    W = synth.normal_bf16((V_high, d), 0.02, seed=d + M, device=dev)
    H = synth.normal_bf16((M, d), 1.0, seed=d + M + 1, device=dev)
    t2f = synth.rank_permutation(2 * V_high, V_high)[:V_high].to(dev)
    ids = Guarded((M, k), torch.int32, dev)
    probs = Guarded((M, k), torch.float32, dev)
    logits = Guarded((M, V_high), torch.float32, dev)
    ws = ws_for("head", dev, M=M, k=k, V_high=V_high)
    vt.draft_head(H, W, t2f, k, out_ids=ids.t, out_probs=probs.t,
                  out_logits=logits.t, ws=ws.t, sample=sample, seed=3,
                  offset=1, check=True)
    for g, name in ((ids, "ids"), (probs, "probs"), (logits, "logits"),
                    (ws, "ws")):
        g.check(name)
    if not sample:
        Hh, Wh, t2f_h = bits_host(H), bits_host(W), t2f.cpu().numpy()
        ref, ref_logits = oracle_head(Hh, Wh, t2f_h, k)
        check_topk(ids.t.cpu().numpy(), probs.t.cpu().numpy(), ref_logits,
                   t2f_h, ref, k)
    # and without the logits output (the tensor-core path keeps them in
    # the workspace instead)
    ids2 = Guarded((M, k), torch.int32, dev)
    probs2 = Guarded((M, k), torch.float32, dev)
    vt.draft_head(H, W, t2f, k, out_ids=ids2.t, out_probs=probs2.t, ws=ws.t,
                  sample=sample, seed=3, offset=1, check=True)
    ids2.check("ids (no logits)")
    probs2.check("probs (no logits)")
    ws.check("ws (no logits)")
    assert torch.equal(ids2.t, ids.t)


@pytest.mark.parametrize("V,V_high,M", [
    (5003, 1111, 3),      # V % 4 != 0: f2t read by each thread
    (20001, 3001, 7),
    (20004, 3001, 7),     # f2t through the shared-memory ring, ragged last chunk
    (128256, 32768, 2),   # the Llama-3-8B shape (ring)
])
def test_draft_q_bounds(V, V_high, M):
    dev = need_cuda()
    logits = torch.from_numpy(np.random.default_rng(V).normal(0, 2, (M, V_high))
                              .astype(np.float32)).to(dev)
    t2f_h = synth.rank_permutation(V, V)[:V_high].numpy()
    f2t_h = np.full(V, -1, np.int32)
    f2t_h[t2f_h] = np.arange(V_high, dtype=np.int32)
    q = Guarded((M, V), torch.float32, dev)
    ws = Guarded((vt.workspace_bytes("q", M=M),), torch.uint8, dev, fill=0)
    vt.draft_q(logits, torch.from_numpy(f2t_h).to(dev), V, temperature=0.9,
               out=q.t, ws=ws.t)
    q.check("q")
    ws.check("ws")
    got = q.t.cpu().numpy()
    s = logits.cpu().numpy().astype(np.float64) / 0.9
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    want = np.zeros((M, V))
    want[:, t2f_h] = p
    assert np.abs(got - want).max() <= 1e-4


def test_draft_head_sets_bounds():
    dev = need_cuda()
    d, V, M, k = 264, 9000, 11, 6
    sizes = (3001, 777)
    Ws = [synth.normal_bf16((n, d), 0.05, seed=800 + n, device=dev) for n in sizes]
    Ts = [synth.rank_permutation(V, 810 + n)[:n].to(dev) for n in sizes]
    H = synth.normal_bf16((M, d), 1.0, seed=820, device=dev)
    sor = np.random.default_rng(821).integers(0, 2, M)
    ids = Guarded((M, k), torch.int32, dev)
    probs = Guarded((M, k), torch.float32, dev)
    V_arr = (ctypes.c_int32 * 2)(*sizes)
    nbytes = vt.load().vt_draft_head_sets_workspace_size(M, d, k, 2, V_arr)
    ws = Guarded((nbytes,), torch.uint8, dev, fill=0)
    vt.draft_head_sets(H, sor, Ws, Ts, k, out_ids=ids.t, out_probs=probs.t,
                       ws=ws.t, check=True)
    for g, name in ((ids, "ids"), (probs, "probs"), (ws, "ws")):
        g.check(name)
    Hh = bits_host(H)
    for s_ in range(2):
        rows = np.nonzero(sor == s_)[0]
        Wh, t2f_h = bits_host(Ws[s_]), Ts[s_].cpu().numpy()
        ref = oracle.draft_head(Hh[rows], Wh, t2f_h, k)
        check_topk(ids.t.cpu().numpy()[rows], probs.t.cpu().numpy()[rows],
                   oracle.head_logits(Hh[rows], Wh), t2f_h, ref, k)


def test_draft_noise_bounds():
    dev = need_cuda()
    full_ids = torch.arange(3001, dtype=torch.int32, device=dev)
    out = Guarded((3001,), torch.float32, dev)
    vt.draft_noise(5, 6, 7, full_ids, out=out.t)
    out.check("noise")
    np.testing.assert_allclose(out.t.cpu().numpy(),
                               oracle.gumbel_noise(5, 6, 7, np.arange(3001)),
                               rtol=2e-6, atol=2e-6)
