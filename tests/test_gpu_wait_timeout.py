"""The failure path of the library's bounded device waits, on the GPU.

vt_selftest_wait_timeout runs the mbarrier wait that the head kernels use
(TMA stages, MMA completion, accumulator hand-over, the final merge's bulk
copy) on a barrier that nothing arrives on: the wait must give up within
its budget, write VT_ERR_TIMEOUT to the error word, and leave the context
usable (a head call afterwards still matches its own result from before).
The same call then plants VT_ERR_TIMEOUT in the error word of a real
workspace, so that the ways a caller learns of it are checked without a
GPU fault: the binding's checked calls raise and clear the word, the host
draft step returns VT_ERR_TIMEOUT and clears it, and the selection clears
its own word when it starts."""
import time

import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import synth
from gpu_util import need_cuda

pytestmark = pytest.mark.gpu

VT_ERR_TIMEOUT = 5


def test_bounded_wait_gives_up_and_reports():
    dev = need_cuda()
    lib = vt.load()
    W = synth.normal_bf16((3000, 256), 0.02, seed=41, device=dev)
    H = synth.normal_bf16((1, 256), 1.0, seed=42, device=dev)
    ids0, probs0 = vt.draft_head(H, W, None, 8)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.vt_selftest_wait_timeout(err.data_ptr(), 2_000_000,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.vt_last_error()
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(err.item()) == VT_ERR_TIMEOUT
    ids1, probs1 = vt.draft_head(H, W, None, 8)
    torch.cuda.synchronize()
    assert torch.equal(ids0, ids1)
    # (the GEMV deals its last rows dynamically, so the softmax sums may
    # differ in the last bits from call to call)
    assert (probs0 - probs1).abs().max().item() <= 1e-6


def plant_timeout(lib, addr):
    """Writes VT_ERR_TIMEOUT at device address ``addr`` through the bounded
    wait's own failure path (a wait of about 0.1 ms that nothing ends)."""
    rc = lib.vt_selftest_wait_timeout(addr, 200_000,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.vt_last_error()
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [1, 6])
def test_checked_head_call_reports_and_clears_the_error_word(M):
    dev = need_cuda()
    lib = vt.load()
    W = synth.normal_bf16((5000, 512), 0.02, seed=43, device=dev)
    H = synth.normal_bf16((M, 512), 1.0, seed=44, device=dev)
    ws = torch.zeros(vt.workspace_bytes("head", M=M, k=8, V_high=5000),
                     dtype=torch.uint8, device=dev)
    ids0, probs0 = vt.draft_head(H, W, None, 8, ws=ws, check=True)
    plant_timeout(lib, ws.data_ptr() + 128)
    with pytest.raises(vt.VTError) as e:
        vt.draft_head(H, W, None, 8, ws=ws, check=True)
    assert e.value.status == VT_ERR_TIMEOUT
    assert int(ws[128:132].view(torch.int32).item()) == 0
    ids1, probs1 = vt.draft_head(H, W, None, 8, ws=ws, check=True)
    assert torch.equal(ids0, ids1)
    # drawing goes through vt_draft_head_ex and is checked the same way
    plant_timeout(lib, ws.data_ptr() + 128)
    with pytest.raises(vt.VTError):
        vt.draft_head(H, W, None, 8, ws=ws, sample=True, seed=1, check=True)


@pytest.mark.parametrize("M", [1, 5])
def test_host_step_returns_timeout_and_recovers(M):
    dev = need_cuda()
    lib = vt.load()
    W = synth.normal_bf16((6000, 1024), 0.02, seed=45, device=dev)
    t2f = synth.rank_permutation(12000, 46)[:6000].to(dev)
    head = vt.HostDraftHead(W, t2f, 10, M)
    H = synth.normal_bf16((M, 1024), 1.0, seed=47)
    ids0 = head(H)[0].clone()
    plant_timeout(lib, head.error_word)
    with pytest.raises(vt.VTError) as e:
        head(H)
    assert e.value.status == VT_ERR_TIMEOUT
    ids1 = head(H)[0]  # the step cleared the word
    assert torch.equal(ids0, ids1)


def test_selection_clears_its_error_word_when_it_starts():
    dev = need_cuda()
    lib = vt.load()
    c = np.random.default_rng(48).integers(0, 1000, 5000).astype(np.uint32)
    counts = torch.from_numpy(c.view(np.int32)).to(dev).view(torch.uint32)
    ws = torch.empty(vt.workspace_bytes("select", V=5000), dtype=torch.uint8,
                     device=dev)
    plant_timeout(lib, ws.data_ptr() + 128)
    t2f, f2t, sums = vt.select_vocab(counts, 700, ws=ws, check=True)
    order = np.lexsort((np.arange(5000), -c.astype(np.int64)))[:700]
    assert t2f.cpu().numpy().tolist() == order.tolist()
