"""vt_draft_head_noalloc: the draft head for callers that cannot allocate.

Callers that may not allocate device memory where they run a draft step
(inside a stream capture that must not gain allocation nodes, on hosts that
forbid allocation after start-up, or as plugins confined to someone else's
memory pool) use this entry point; it keeps its scratch in a fixed device
array inside the library instead of taking a workspace.  These tests call
it through the C ABI on two calls in a row and check each call against
vt_draft_head (the entry point with a caller-provided workspace) within the
tolerances of the other head tests, and its top-k against the oracle by
the rule of the other head tests (ids may differ only where oracle logits
are closer than the logit tolerance).  For M = 1 both entry points run the
same kernel, so their ids must be equal.  The file sorts last so that a
run that stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle
import synth
from gpu_util import (LOGIT_RTOL, PROB_ATOL, bits_host, check_logits,
                      check_topk, need_cuda)

pytestmark = pytest.mark.gpu

VT_OK, VT_ERR_UNSUPPORTED = 0, 3


def noalloc_fn():
    lib = vt.load()
    fn = lib.vt_draft_head_noalloc
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [p, i32, i32, i64, p, i32, p, i32, p, p, p, p]
    fn.restype = ctypes.c_int
    return lib, fn


def run_noalloc(fn, H, W_high, t2f, k):
    M, d = H.shape
    V_high = W_high.shape[0]
    ids = torch.full((M, k), -7, dtype=torch.int32, device=H.device)
    probs = torch.full((M, k), -1.0, dtype=torch.float32, device=H.device)
    logits = torch.full((M, V_high), float("nan"), dtype=torch.float32,
                        device=H.device)
    rc = fn(H.data_ptr(), M, d, H.stride(0), W_high.data_ptr(), V_high,
            None if t2f is None else t2f.data_ptr(), k, ids.data_ptr(),
            probs.data_ptr(), logits.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    return rc, ids, probs, logits


@pytest.mark.parametrize("d,V,V_high,M,k", [
    (4096, 128256, 32768, 1, 10),   # the Llama-3-8B-shaped draft step
    (1032, 9000, 5000, 6, 8),       # two groups of hidden states, ragged d
])
def test_noalloc_matches_workspace_entry_point(d, V, V_high, M, k):
    dev = need_cuda()
    lib, fn = noalloc_fn()
    W_high = synth.normal_bf16((V_high, d), 0.02, seed=31, device=dev)
    H = synth.normal_bf16((M, d), 1.0, seed=32, device=dev)
    t2f = synth.rank_permutation(V, 33)[:V_high].to(dev)
    ref_logits = torch.empty(M, V_high, dtype=torch.float32, device=dev)
    ref_ids, ref_probs = vt.draft_head(H, W_high, t2f, k, out_logits=ref_logits)
    Hh, Wh, t2f_h = bits_host(H), bits_host(W_high), t2f.cpu().numpy()
    o_ref = oracle.draft_head(Hh, Wh, t2f_h, k)
    o_logits = oracle.head_logits(Hh, Wh)
    for call in range(2):  # two calls in a row share the same scratch
        rc, ids, probs, logits = run_noalloc(fn, H, W_high, t2f, k)
        assert rc == VT_OK, lib.vt_last_error()
        torch.cuda.synchronize()
        # against the workspace entry point: same results within tolerance
        tol = LOGIT_RTOL * (1.0 + ref_logits.abs())
        assert ((logits - ref_logits).abs() <= tol).all(), f"call {call}"
        assert (probs - ref_probs).abs().max().item() <= PROB_ATOL
        if M == 1:  # the same GEMV kernel: the same ids
            assert torch.equal(ids, ref_ids), f"call {call}: ids differ"
        # against the oracle
        check_logits(logits.cpu().numpy(), o_logits)
        check_topk(ids.cpu().numpy(), probs.cpu().numpy(), o_logits, t2f_h,
                   o_ref, k)


def test_noalloc_rejects_scratch_beyond_its_limit():
    """M >= 4 with k = 32 needs more than the fixed 1 MiB of scratch."""
    dev = need_cuda()
    lib, fn = noalloc_fn()
    W_high = torch.zeros(64, 256, dtype=torch.bfloat16, device=dev)
    H = torch.zeros(4, 256, dtype=torch.bfloat16, device=dev)
    rc, _, _, _ = run_noalloc(fn, H, W_high, None, 32)
    assert rc == VT_ERR_UNSUPPORTED
    assert b"scratch" in lib.vt_last_error()
