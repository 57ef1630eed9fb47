"""ctypes front end of the plain CPU oracle (``oracle.cpp``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The CUDA library under ``frequency_ranked_drafter_gb300/``
never imports, links or executes it, and this package imports nothing from
that library.

The functions take and return numpy arrays.  bf16 tensors are passed as their
raw ``uint16`` bit patterns, so the oracle and the CUDA path read the very
same bytes.  Sources are cited in ``oracle.cpp`` beside each step.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force on tiny inputs, library routines on special cases, closed forms
and invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``_build/liboracle.so`` (g++, -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # A test may point this at a deliberately broken build of the same
        # source to check that the pins catch the mistake.
        override = os.environ.get("FRD_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        p = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_count_tokens.argtypes = [p, i64, i32, p, p]
        lib.oracle_select_vocab.argtypes = [p, i32, i32, p, p, p, p, p]
        lib.oracle_gather_rows.argtypes = [p, i64, i32, p, i32, p]
        lib.oracle_head_logits.argtypes = [p, i32, i32, i64, p, i32, p]
        lib.oracle_draft_head.argtypes = [p, i32, i32, i64, p, i32, p, i32,
                                          p, p, p, p, p, p]
        u64, f64 = ctypes.c_uint64, ctypes.c_double
        lib.oracle_philox4x32_10.argtypes = [p, p, p]
        lib.oracle_gather_bias.argtypes = [p, i64, p, i32, p]
        lib.oracle_draft_q.argtypes = [p, i32, i32, i64, p, i32, p, p, f64,
                                       i32, p]
        lib.oracle_draft_q.restype = ctypes.c_int
        lib.oracle_gather_bias.restype = i64
        lib.oracle_gumbel_noise.argtypes = [u64, u64, i32, p, i64, p]
        lib.oracle_draft_head_ex.argtypes = [p, i32, i32, i64, p, i32, p, p,
                                             f64, i32, u64, u64, i32, i32, p,
                                             p, p, p, p, p, p]
        for fn in (lib.oracle_count_tokens, lib.oracle_select_vocab,
                   lib.oracle_gather_rows, lib.oracle_head_logits,
                   lib.oracle_draft_head, lib.oracle_philox4x32_10,
                   lib.oracle_gumbel_noise, lib.oracle_draft_head_ex):
            fn.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    """bf16 bit patterns as a contiguous uint16 array."""
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return np.ascontiguousarray(a)


def count_tokens(tokens, V: int):
    """Histogram of ``tokens`` over ids 0..V-1 -> (counts uint64[V], n_invalid)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    counts = np.zeros(V, dtype=np.uint64)
    n_invalid = np.zeros(1, dtype=np.uint64)
    rc = _load().oracle_count_tokens(_ptr(tokens), tokens.size, V,
                                     _ptr(counts), _ptr(n_invalid))
    if rc:
        raise ValueError(f"oracle_count_tokens: bad arguments (rc={rc})")
    return counts, int(n_invalid[0])


def select_vocab(counts, V_high: int):
    """Top-V_high selection -> dict(t2f, f2t, kept, total, coverage)."""
    counts = np.ascontiguousarray(counts, dtype=np.uint64)
    V = counts.size
    t2f = np.empty(V_high, dtype=np.int32)
    f2t = np.empty(V, dtype=np.int32)
    kept = np.zeros(1, dtype=np.uint64)
    total = np.zeros(1, dtype=np.uint64)
    cov = np.zeros(1, dtype=np.float64)
    rc = _load().oracle_select_vocab(_ptr(counts), V, V_high, _ptr(t2f),
                                     _ptr(f2t), _ptr(kept), _ptr(total),
                                     _ptr(cov))
    if rc:
        raise ValueError(f"oracle_select_vocab: bad arguments (rc={rc})")
    return dict(t2f=t2f, f2t=f2t, kept=int(kept[0]), total=int(total[0]),
                coverage=float(cov[0]))


def gather_rows(W, t2f):
    """W_high[i] = W[t2f[i]] on bf16 bit patterns -> (W_high, n_bad_rows_flag)."""
    W = _u16(W)
    V, d = W.shape
    t2f = np.ascontiguousarray(t2f, dtype=np.int32)
    out = np.empty((t2f.size, d), dtype=np.uint16)
    rc = _load().oracle_gather_rows(_ptr(W), V, d, _ptr(t2f), t2f.size,
                                    _ptr(out))
    return out, rc


def gather_bias(b, t2f):
    """b_high[i] = b[t2f[i]] (fp32) -> (b_high, number of ids out of range)."""
    b = np.ascontiguousarray(b, dtype=np.float32)
    t2f = np.ascontiguousarray(t2f, dtype=np.int32)
    out = np.empty(t2f.size, dtype=np.float32)
    bad = _load().oracle_gather_bias(_ptr(b), b.size, _ptr(t2f), t2f.size,
                                     _ptr(out))
    return out, int(bad)


def head_logits(H, W_high):
    """fp64 logits[M, V_high] = H . W_high^T from bf16 bit patterns."""
    H = _u16(H)
    W_high = _u16(W_high)
    M, d = H.shape
    V_high, d2 = W_high.shape
    assert d == d2
    out = np.empty((M, V_high), dtype=np.float64)
    _load().oracle_head_logits(_ptr(H), M, d, d, _ptr(W_high), V_high,
                               _ptr(out))
    return out


def draft_head(H, W_high, t2f, k: int):
    """Trimmed head step: logits -> softmax over V_high -> top-k -> remap.

    Returns dict with ids[M,k] (full vocabulary), probs[M,k], logits[M,k],
    trimmed[M,k], row_max[M], row_sumexp[M]; ``t2f=None`` is the identity.
    """
    H = _u16(H)
    W_high = _u16(W_high)
    M, d = H.shape
    V_high = W_high.shape[0]
    if t2f is not None:
        t2f = np.ascontiguousarray(t2f, dtype=np.int32)
        assert t2f.size == V_high
    ids = np.empty((M, k), dtype=np.int32)
    probs = np.empty((M, k), dtype=np.float64)
    logits = np.empty((M, k), dtype=np.float64)
    trimmed = np.empty((M, k), dtype=np.int32)
    rmax = np.empty(M, dtype=np.float64)
    rsum = np.empty(M, dtype=np.float64)
    rc = _load().oracle_draft_head(_ptr(H), M, d, d, _ptr(W_high), V_high,
                                   _ptr(t2f), k, _ptr(ids), _ptr(probs),
                                   _ptr(logits), _ptr(trimmed), _ptr(rmax),
                                   _ptr(rsum))
    if rc:
        raise ValueError(f"oracle_draft_head: bad arguments (rc={rc})")
    return dict(ids=ids, probs=probs, logits=logits, trimmed=trimmed,
                row_max=rmax, row_sumexp=rsum)


def philox4x32_10(ctr, key):
    """Philox4x32-10 output block (4 x uint32) for counter[4], key[2]."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    kk = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(kk), _ptr(out))
    return out


def gumbel_noise(seed: int, offset: int, m: int, full_ids):
    """Gumbel noise of the given full ids for hidden state m at (seed, offset)."""
    f = np.ascontiguousarray(full_ids, dtype=np.int32)
    out = np.empty(f.size, dtype=np.float64)
    _load().oracle_gumbel_noise(ctypes.c_uint64(seed), ctypes.c_uint64(offset),
                                m, _ptr(f), f.size, _ptr(out))
    return out


def draft_head_ex(H, W_high, t2f, k: int, bias=None, temperature=1.0,
                  sample=False, seed=0, offset=0, m_base=0):
    """Draft step with options: optional kept-row bias (fp32), temperature,
    top-k or Gumbel-max sampling (k draws without replacement); the noise of
    row j uses hidden-state index m_base + j.

    Returns dict with ids[M,k], probs[M,k], scores[M,k] (selection keys),
    logits[M,k], trimmed[M,k], row_max[M] (of logit/T), row_sumexp[M].
    """
    H = _u16(H)
    W_high = _u16(W_high)
    M, d = H.shape
    V_high = W_high.shape[0]
    if t2f is not None:
        t2f = np.ascontiguousarray(t2f, dtype=np.int32)
        assert t2f.size == V_high
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        assert bias.size == V_high
    ids = np.empty((M, k), dtype=np.int32)
    probs = np.empty((M, k), dtype=np.float64)
    scores = np.empty((M, k), dtype=np.float64)
    logits = np.empty((M, k), dtype=np.float64)
    trimmed = np.empty((M, k), dtype=np.int32)
    rmax = np.empty(M, dtype=np.float64)
    rsum = np.empty(M, dtype=np.float64)
    rc = _load().oracle_draft_head_ex(
        _ptr(H), M, d, d, _ptr(W_high), V_high, _ptr(t2f), _ptr(bias),
        ctypes.c_double(temperature), 1 if sample else 0,
        ctypes.c_uint64(seed), ctypes.c_uint64(offset), m_base, k, _ptr(ids),
        _ptr(probs), _ptr(scores), _ptr(logits), _ptr(trimmed), _ptr(rmax),
        _ptr(rsum))
    if rc:
        raise ValueError(f"oracle_draft_head_ex: bad arguments (rc={rc})")
    return dict(ids=ids, probs=probs, scores=scores, logits=logits,
                trimmed=trimmed, row_max=rmax, row_sumexp=rsum)


def draft_q(H, W_high, t2f, V: int, bias=None, temperature=1.0):
    """Full-vocabulary draft distribution q[M, V]: the trimmed softmax at the
    kept ids (through t2f), 0 at dropped ids."""
    H = _u16(H)
    W_high = _u16(W_high)
    M, d = H.shape
    V_high = W_high.shape[0]
    if t2f is not None:
        t2f = np.ascontiguousarray(t2f, dtype=np.int32)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
    q = np.empty((M, V), dtype=np.float64)
    rc = _load().oracle_draft_q(_ptr(H), M, d, d, _ptr(W_high), V_high,
                                _ptr(t2f), _ptr(bias),
                                ctypes.c_double(temperature), V, _ptr(q))
    if rc:
        raise ValueError(f"oracle_draft_q: bad arguments (rc={rc})")
    return q
