"""The failure path of the library's bounded device waits, on the GPU.

vt_selftest_wait_timeout runs the mbarrier wait that the head kernels use
(TMA stages, MMA completion, accumulator hand-over, the final merge's bulk
copy) on a barrier that nothing arrives on: the wait must give up within
its budget, write VT_ERR_TIMEOUT to the error word, and leave the context
usable (a head call afterwards still matches its own result from before)."""
import time

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
    assert torch.equal(probs0, probs1)
