"""The C ABI without a GPU: the library builds and loads, exports every
function include/vt.h declares, and rejects bad arguments on the host
before touching the device (nothing here makes a CUDA call)."""
import ctypes
import os
import re

import pytest

import frequency_ranked_drafter_gb300 as vt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vt.h")

OK, INVALID, CUDA, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3, 4
FAKE = 1 << 20  # a 256-byte aligned non-null address never dereferenced


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vt_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return vt.load()


def test_header_declares_the_four_calls():
    names = declared_functions()
    for fn in ("vt_count_tokens", "vt_select_vocab", "vt_gather_rows",
               "vt_draft_head"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(vt.library_path())
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_release_build_has_no_checks(lib):
    assert lib.vt_debug_build() == 0
    assert lib.vt_debug_checks() == 0  # no check words: no device access
    assert lib.vt_selftest_check(None, 10, None) == INVALID
    assert lib.vt_selftest_check(FAKE, 0, None) == INVALID
    assert lib.vt_selftest_check(FAKE + 2, 10, None) == INVALID


def test_checked_build_compiles_and_exports_the_same_symbols():
    """The bounds-checked variant (-DVT_CHECKS) builds, says so, and exports
    every function vt.h declares."""
    from frequency_ranked_drafter_gb300 import build as vt_build
    path = vt_build.build(checks=True)
    raw = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing
    raw.vt_debug_build.restype = ctypes.c_int
    assert raw.vt_debug_build() == 1


def test_status_strings_and_version(lib):
    assert lib.vt_status_string(0) == b"VT_OK"
    assert lib.vt_status_string(1) == b"VT_ERR_INVALID_ARG"
    assert lib.vt_status_string(99) == b"VT_ERR_UNKNOWN"
    assert lib.vt_version() >= 100


def test_workspace_sizes(lib):
    assert lib.vt_count_tokens_workspace_size(0) == 0
    assert lib.vt_count_tokens_workspace_size(128256) >= 128256
    assert lib.vt_select_vocab_workspace_size(128256) >= 16 * 128256
    assert lib.vt_draft_head_workspace_size(1, 32768, 10) > 256
    # the tensor-core path (M >= 2) keeps the [M, V_high] fp32 logits
    assert lib.vt_draft_head_workspace_size(64, 32768, 10) >= 64 * 32768 * 4
    assert lib.vt_draft_head_workspace_size(0, 32768, 10) == 0


def test_workspace_size_dispatcher_matches_the_per_op_functions(lib):
    """vt_workspace_size(op, M, n, k) returns what each operation's own size
    function returns (n is V for the histogram and the selection, V_high for
    the head), and 0 for an unknown op."""
    COUNT, SELECT, HEAD, Q = 0, 1, 2, 3
    for V in (1, 4096, 128256, 300000):
        assert lib.vt_workspace_size(COUNT, 0, V, 0) == \
            lib.vt_count_tokens_workspace_size(V)
        assert lib.vt_workspace_size(SELECT, 7, V, 3) == \
            lib.vt_select_vocab_workspace_size(V)
    for M, V_high, k in ((1, 32768, 10), (4, 1000, 32), (60, 8192, 10),
                         (256, 128256, 1), (0, 10, 1)):
        assert lib.vt_workspace_size(HEAD, M, V_high, k) == \
            lib.vt_draft_head_workspace_size(M, V_high, k)
        assert lib.vt_workspace_size(Q, M, 0, 0) == \
            lib.vt_draft_q_workspace_size(M)
    assert lib.vt_workspace_size(4, 1, 1, 1) == 0
    assert lib.vt_workspace_size(-1, 1, 1, 1) == 0
    assert vt.workspace_bytes("head", M=60, V_high=8192, k=10) == \
        lib.vt_draft_head_workspace_size(60, 8192, 10)


def test_workspaces_hold_the_error_word_at_byte_128(lib):
    """Every workspace that has an error word keeps it at byte 128, so
    workspaces are at least 132 bytes."""
    assert lib.vt_select_vocab_workspace_size(1) >= 132
    assert lib.vt_draft_head_workspace_size(1, 1, 1) >= 132
    assert lib.vt_draft_head_workspace_size(2, 1, 1) >= 132


def test_host_step_error_word_of_null_handle(lib):
    assert lib.vt_host_step_error_word(None) is None


def test_draft_head_rejects_bad_arguments(lib):
    ws_ok = lib.vt_draft_head_workspace_size(1, 32768, 10)

    def call(H=FAKE, M=1, d=4096, ldh=4096, W=FAKE, V_high=32768, t2f=None,
             k=10, ids=FAKE, probs=FAKE, logits=None, ws=FAKE, ws_bytes=ws_ok):
        return lib.vt_draft_head(H, M, d, ldh, W, V_high, t2f, k, ids, probs,
                                 logits, ws, ws_bytes, None)

    assert call(H=None) == INVALID
    assert call(M=0) == INVALID
    assert call(M=257) == INVALID
    assert call(d=4095, ldh=4095) == INVALID
    assert call(ldh=4000) == INVALID
    assert call(k=0) == INVALID
    assert call(k=33) == INVALID
    assert call(V_high=5, k=6) == INVALID
    assert call(H=FAKE + 2) == INVALID  # misaligned
    assert call(ws=None) == WORKSPACE
    assert call(ws_bytes=ws_ok - 1) == WORKSPACE
    assert call(ws=FAKE + 16) == WORKSPACE
    assert b"workspace" in lib.vt_last_error()


def test_count_select_gather_reject_bad_arguments(lib):
    wsc = lib.vt_count_tokens_workspace_size(100)
    assert lib.vt_count_tokens(FAKE, 10, 0, FAKE, None, FAKE, wsc, None) == INVALID
    assert lib.vt_count_tokens(FAKE, -1, 100, FAKE, None, FAKE, wsc, None) == INVALID
    assert lib.vt_count_tokens(FAKE + 4, 10, 100, FAKE, None, FAKE, wsc, None) == INVALID
    assert lib.vt_count_tokens(FAKE, 10, 100, FAKE, None, FAKE, wsc - 1, None) == WORKSPACE
    # n == 0 is a valid no-op that never touches the device
    assert lib.vt_count_tokens(None, 0, 100, FAKE, None, FAKE, wsc, None) == OK

    wss = lib.vt_select_vocab_workspace_size(100)
    assert lib.vt_select_vocab(FAKE, 100, 0, FAKE, FAKE, FAKE, FAKE, wss, None) == INVALID
    assert lib.vt_select_vocab(FAKE, 100, 101, FAKE, FAKE, FAKE, FAKE, wss, None) == INVALID
    assert lib.vt_select_vocab(FAKE, 100, 10, FAKE, FAKE, FAKE, FAKE, wss - 1, None) == WORKSPACE
    assert lib.vt_select_vocab(FAKE, 1 << 25, 10, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == UNSUPPORTED

    assert lib.vt_gather_rows(FAKE, 100, 12, FAKE, 10, FAKE * 4, None, None) == INVALID
    assert lib.vt_gather_rows(FAKE, 100, 16, None, 10, FAKE * 4, None, None) == INVALID
    # overlapping output
    assert lib.vt_gather_rows(FAKE, 100, 16, FAKE, 10, FAKE + 32, None, None) == INVALID


def test_python_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(TypeError):
        vt.count_tokens(torch.zeros(8, dtype=torch.int32), 4)
    with pytest.raises(TypeError):
        vt.draft_head(torch.zeros(1, 8, dtype=torch.bfloat16),
                      torch.zeros(4, 8, dtype=torch.bfloat16), None, 1)


def test_draft_head_ex_rejects_bad_options(lib):
    """Temperature must be finite and positive, the mode known, the bias
    4-byte aligned; all checked on the host, nothing launched."""
    ws_ok = lib.vt_draft_head_workspace_size(1, 4096, 10)

    def call(opts):
        return lib.vt_draft_head_ex(FAKE, 1, 256, 256, FAKE, 4096, None, 10,
                                    ctypes.byref(opts) if opts else None,
                                    FAKE, FAKE, None, FAKE, ws_ok, None)

    bad = [vt.HeadOptions(None, 0.0, 0, 0, 0),
           vt.HeadOptions(None, -1.0, 0, 0, 0),
           vt.HeadOptions(None, float("nan"), 0, 0, 0),
           vt.HeadOptions(None, float("inf"), 1, 0, 0),
           vt.HeadOptions(None, 1.0, 2, 0, 0),
           vt.HeadOptions(FAKE + 2, 1.0, 0, 0, 0)]
    for opts in bad:
        assert call(opts) == INVALID
    # the head's own argument checks still apply under options
    opts = vt.HeadOptions(None, 1.0, 1, 7, 0)
    assert lib.vt_draft_head_ex(FAKE, 1, 256, 256, FAKE, 4096, None, 0,
                                ctypes.byref(opts), FAKE, FAKE, None, FAKE,
                                ws_ok, None) == INVALID
    assert lib.vt_draft_head_ex(FAKE, 1, 256, 256, FAKE, 4096, None, 10,
                                ctypes.byref(opts), FAKE, FAKE, None, FAKE,
                                ws_ok - 16, None) == WORKSPACE


def test_draft_noise_rejects_bad_arguments(lib):
    assert lib.vt_draft_noise(1, 2, 0, FAKE, -1, FAKE, None) == INVALID
    assert lib.vt_draft_noise(1, 2, -1, FAKE, 5, FAKE, None) == INVALID
    assert lib.vt_draft_noise(1, 2, 0, None, 5, FAKE, None) == INVALID
    assert lib.vt_draft_noise(1, 2, 0, None, 0, None, None) == OK


def test_gather_bias_rejects_bad_arguments(lib):
    assert lib.vt_gather_bias(None, 10, FAKE, 5, FAKE, None, None) == INVALID
    assert lib.vt_gather_bias(FAKE, 0, FAKE, 5, FAKE + 4096, None, None) == INVALID
    assert lib.vt_gather_bias(FAKE + 2, 10, FAKE, 5, FAKE + 4096, None, None) == INVALID
    # b_high overlapping b
    assert lib.vt_gather_bias(FAKE, 100, FAKE + 8192, 50, FAKE + 40, None,
                              None) == INVALID


def test_draft_q_rejects_bad_arguments(lib):
    ws = lib.vt_draft_q_workspace_size(4)
    assert ws == 32 and lib.vt_draft_q_workspace_size(0) == 0
    good = dict(logits=FAKE, M=4, V_high=100, f2t=FAKE + 65536, V=500, T=1.0,
                q=FAKE + 131072, ws=FAKE + 262144, nbytes=ws)

    def call(**kw):
        a = dict(good, **kw)
        return lib.vt_draft_q(a["logits"], a["M"], a["V_high"], a["f2t"], a["V"],
                              a["T"], a["q"], a["ws"], a["nbytes"], None)

    assert call(logits=None) == INVALID
    assert call(M=0) == INVALID
    assert call(V=99) == INVALID
    assert call(f2t=None) == INVALID          # identity needs V == V_high
    assert call(T=0.0) == INVALID
    assert call(T=float("nan")) == INVALID
    assert call(q=FAKE + 2) == INVALID        # misaligned and overlapping
    assert call(q=FAKE + 400) == INVALID      # overlaps logits
    assert call(nbytes=ws - 8) == WORKSPACE
    assert call(ws=None) == WORKSPACE


def test_draft_head_sets_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    W = (P * 2)(FAKE, FAKE + 1 << 24)
    V = (ctypes.c_int32 * 2)(100, 200)
    sor = (ctypes.c_int32 * 3)(0, 1, 0)
    ws = lib.vt_draft_head_sets_workspace_size(3, 64, 5, 2, V)
    assert ws > 0 and lib.vt_draft_head_sets_workspace_size(3, 64, 5, 0, V) == 0

    def call(sor=sor, S=2, W=W, V=V, k=5, opts=None, nbytes=ws):
        return lib.vt_draft_head_sets(FAKE, 3, 64, 64, sor, S, W, V, None, None,
                                      k, ctypes.byref(opts) if opts else None,
                                      FAKE, FAKE, FAKE, nbytes, None)

    assert call(sor=(ctypes.c_int32 * 3)(0, 2, 0)) == INVALID   # set out of range
    assert call(V=(ctypes.c_int32 * 2)(100, 3)) == INVALID      # V_high < k
    assert call(W=(P * 2)(FAKE, FAKE + 8)) == INVALID           # misaligned W
    assert call(opts=vt.HeadOptions(FAKE, 1.0, 0, 0, 0)) == INVALID  # bias in opts
    assert call(nbytes=ws - 256) == WORKSPACE


def test_host_step_rejects_bad_arguments(lib):
    """Checked before anything is allocated: no handle, drawing, bad sizes."""
    h = ctypes.c_void_p()
    assert lib.vt_host_step_create(FAKE, 1000, 256, None, 1, 10, None, None) == INVALID
    draw = vt.HeadOptions(None, 1.0, 1, 0, 0)
    assert lib.vt_host_step_create(FAKE, 1000, 256, None, 1, 10, ctypes.byref(draw),
                                   ctypes.byref(h)) == INVALID
    assert lib.vt_host_step_create(FAKE, 5, 256, None, 1, 10, None,
                                   ctypes.byref(h)) == INVALID   # V_high < k
    assert lib.vt_host_step_create(FAKE, 1000, 250, None, 1, 10, None,
                                   ctypes.byref(h)) == INVALID   # d % 8
    assert not h.value
    assert lib.vt_host_step_run(None, FAKE, FAKE, FAKE) == INVALID
    lib.vt_host_step_destroy(None)


def test_selftest_wait_timeout_rejects_bad_arguments(lib):
    """Checked on the host, nothing launched: no error word, a misaligned
    one, and budgets outside 1 .. 2^31 cycles."""
    assert lib.vt_selftest_wait_timeout(None, 1000, None) == INVALID
    assert lib.vt_selftest_wait_timeout(FAKE + 2, 1000, None) == INVALID
    assert lib.vt_selftest_wait_timeout(FAKE, 0, None) == INVALID
    assert lib.vt_selftest_wait_timeout(FAKE, (1 << 31) + 1, None) == INVALID
    assert b"budget" in lib.vt_last_error()
