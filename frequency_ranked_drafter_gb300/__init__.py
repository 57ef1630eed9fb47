"""GB300-native frequency-ranked trimmed drafter head (VocabTrim / FR-Spec).

A thin ctypes binding over the C ABI of ``include/vt.h``.  Every step of the
path runs in the library's CUDA kernels; this module only checks tensor
types, allocates outputs and workspaces with PyTorch, and passes device
pointers and the current CUDA stream.  There is no CPU fallback: if the
library is missing or a call fails, an exception is raised.

Functions (same names as the C ABI without the ``vt_`` prefix):
  count_tokens(tokens, V)            -> (counts uint32[V], n_invalid)
  select_vocab(counts, V_high)       -> (t2f, f2t, sums)   sums = [kept, total]
  gather_rows(W, t2f)                -> W_high
  draft_head(H, W_high, t2f, k)      -> (ids int32[M,k], probs f32[M,k])
and the conveniences build_vocab(...) and coverage(sums).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = ["VTError", "load", "library_path", "count_tokens", "select_vocab",
           "gather_rows", "draft_head", "draft_head_host", "build_vocab",
           "coverage", "Workspace", "workspace_bytes", "check_error_word",
           "save_vocab", "load_vocab"]

VT_OK = 0
_STATUS = {0: "VT_OK", 1: "VT_ERR_INVALID_ARG", 2: "VT_ERR_CUDA",
           3: "VT_ERR_UNSUPPORTED", 4: "VT_ERR_WORKSPACE", 5: "VT_ERR_TIMEOUT"}


class VTError(RuntimeError):
    def __init__(self, fn: str, status: int, why: str):
        super().__init__(f"{fn}: {_STATUS.get(status, status)}: {why}")
        self.status = status


_lib = None
_lock = threading.Lock()

VT_HEAD_TOPK, VT_HEAD_SAMPLE = 0, 1


class HeadOptions(ctypes.Structure):
    """``vt_head_options`` of the C ABI."""
    _fields_ = [("bias_high", ctypes.c_void_p), ("temperature", ctypes.c_float),
                ("mode", ctypes.c_int32), ("seed", ctypes.c_uint64),
                ("offset", ctypes.c_uint64)]


def _checked() -> bool:
    """VT_CHECKS=1 in the environment selects the bounds-checked debug build."""
    return os.environ.get("VT_CHECKS", "") == "1"


def library_path() -> str:
    return _build.CHECKS_LIB_PATH if _checked() else _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load (building first if needed) the CUDA library; raises if absent.
    With VT_CHECKS=1 in the environment, the bounds-checked debug build."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        checks = _checked()
        path = library_path()
        if not os.path.exists(path) or not _build.up_to_date(checks):
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {path}")
            _build.build(checks=checks)
        lib = ctypes.CDLL(path)
        p, i32, i64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                           ctypes.c_size_t)
        sig = {
            "vt_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "vt_last_error": ([], ctypes.c_char_p),
            "vt_version": ([], ctypes.c_int),
            "vt_debug_build": ([], ctypes.c_int),
            "vt_debug_checks": ([], ctypes.c_int),
            "vt_count_tokens_workspace_size": ([i32], sz),
            "vt_count_tokens": ([p, i64, i32, p, p, p, sz, p], ctypes.c_int),
            "vt_select_vocab_workspace_size": ([i32], sz),
            "vt_select_vocab": ([p, i32, i32, p, p, p, p, sz, p], ctypes.c_int),
            "vt_gather_rows": ([p, i64, i32, p, i32, p, p, p], ctypes.c_int),
            "vt_gather_bias": ([p, i64, p, i32, p, p, p], ctypes.c_int),
            "vt_draft_head_workspace_size": ([i32, i32, i32], sz),
            "vt_draft_head": ([p, i32, i32, i64, p, i32, p, i32, p, p, p, p,
                               sz, p], ctypes.c_int),
            "vt_draft_head_ex": ([p, i32, i32, i64, p, i32, p, i32,
                                  ctypes.POINTER(HeadOptions), p, p, p, p, sz,
                                  p], ctypes.c_int),
            "vt_selftest_wait_timeout": ([p, i64, p], ctypes.c_int),
            "vt_selftest_check": ([p, i32, p], ctypes.c_int),
            "vt_draft_noise": ([ctypes.c_uint64, ctypes.c_uint64, i32, p, i64,
                                p, p], ctypes.c_int),
            "vt_draft_q_workspace_size": ([i32], sz),
            "vt_host_step_create": ([p, i32, i32, p, i32, i32,
                                     ctypes.POINTER(HeadOptions),
                                     ctypes.POINTER(p)], ctypes.c_int),
            "vt_host_step_run": ([p, p, p, p], ctypes.c_int),
            "vt_host_step_staging": ([p], p),
            "vt_host_step_error_word": ([p], p),
            "vt_workspace_size": ([i32, i32, i32, i32], sz),
            "vt_host_step_destroy": ([p], None),
            "vt_draft_head_sets_workspace_size": ([i32, i32, i32, i32, p], sz),
            "vt_draft_head_sets": ([p, i32, i32, i64, p, i32, p, p, p, p, i32,
                                    ctypes.POINTER(HeadOptions), p, p, p, sz, p],
                                   ctypes.c_int),
            "vt_draft_q": ([p, i32, i32, p, i32, ctypes.c_float, p, p, sz, p],
                           ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != VT_OK:
        why = load().vt_last_error().decode(errors="replace")
        raise VTError(fn, status, why)


VT_ERR_TIMEOUT = 5
_ERR_WORD = 128  # byte offset of the device error word in every workspace


def check_error_word(fn: str, ws: torch.Tensor):
    """Reads the device error word of a call's workspace (synchronising
    with the workspace's device); if it was set, zero-fills the workspace
    (the word, and any counters the interrupted call left set) and raises
    VTError(VT_ERR_TIMEOUT): a bounded wait inside that call's kernels gave
    up, and its outputs are incomplete."""
    word = ws[_ERR_WORD:_ERR_WORD + 4].view(torch.int32)
    e = int(word.item())
    if e != 0:
        ws.zero_()
        raise VTError(fn, e, "a bounded wait inside the kernels gave up; "
                             "the call's outputs are incomplete")


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream(device: torch.device):
    return torch.cuda.current_stream(device).cuda_stream


def _cuda(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class Workspace:
    """Per-device, per-stream scratch buffers, grown on demand.

    The draft-head workspace must start zero-filled; the kernels leave it
    zero-filled again, so it is allocated with zeros once and reused.
    """

    def __init__(self):
        self._bufs: dict = {}

    def get(self, kind: str, nbytes: int, device: torch.device,
            zeroed: bool) -> torch.Tensor:
        key = (kind, device.index, _stream(device))
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < nbytes:
            alloc = torch.zeros if zeroed else torch.empty
            buf = alloc(max(nbytes, 256), dtype=torch.uint8, device=device)
            self._bufs[key] = buf
        return buf


_ws = Workspace()


_OPS = {"count": 0, "select": 1, "head": 2, "q": 3}


def workspace_bytes(op: str, V: int = 0, M: int = 1, k: int = 1,
                    V_high: int = 1) -> int:
    """Workspace size (vt_workspace_size) of op "count" (V), "select" (V),
    "head" (M, V_high, k) or "q" (M)."""
    if op not in _OPS:
        raise ValueError(op)
    n = V if op in ("count", "select") else V_high
    return load().vt_workspace_size(_OPS[op], M, n, k)


def count_tokens(tokens: torch.Tensor, V: int, counts: torch.Tensor | None = None,
                 n_invalid: torch.Tensor | None = None,
                 ws: torch.Tensor | None = None):
    """Histogram of int32 ``tokens`` over ids 0..V-1 (accumulates into
    ``counts`` if given).  Returns (counts uint32[V], n_invalid int64[1])."""
    _cuda(tokens, "tokens", torch.int32)
    dev = tokens.device
    if counts is None:
        counts = torch.zeros(V, dtype=torch.uint32, device=dev)
    _cuda(counts, "counts", torch.uint32)
    if n_invalid is None:
        n_invalid = torch.zeros(1, dtype=torch.int64, device=dev)
    _cuda(n_invalid, "n_invalid", torch.int64)
    lib = load()
    nbytes = lib.vt_count_tokens_workspace_size(V)
    if ws is None:
        ws = _ws.get("count", nbytes, dev, zeroed=False)
    _check("vt_count_tokens", lib.vt_count_tokens(
        _ptr(tokens), tokens.numel(), V, _ptr(counts), _ptr(n_invalid),
        _ptr(ws), ws.numel(), _stream(dev)))
    return counts, n_invalid


def select_vocab(counts: torch.Tensor, V_high: int,
                 ws: torch.Tensor | None = None, out: tuple | None = None,
                 check: bool = False):
    """Top-V_high ids by count (ties: lower id).  Returns (t2f int32[V_high],
    f2t int32[V] with -1 for dropped ids, sums int64[2] = [kept, total]).
    ``check=True`` synchronises and raises VTError(VT_ERR_TIMEOUT) if a
    bounded wait of the selection gave up."""
    _cuda(counts, "counts", torch.uint32)
    dev = counts.device
    V = counts.numel()
    if out is None:
        t2f = torch.empty(V_high, dtype=torch.int32, device=dev)
        f2t = torch.empty(V, dtype=torch.int32, device=dev)
        sums = torch.empty(2, dtype=torch.int64, device=dev)
    else:
        t2f, f2t, sums = out
    lib = load()
    nbytes = lib.vt_select_vocab_workspace_size(V)
    if ws is None:
        ws = _ws.get("select", nbytes, dev, zeroed=False)
    _check("vt_select_vocab", lib.vt_select_vocab(
        _ptr(counts), V, V_high, _ptr(t2f), _ptr(f2t), _ptr(sums), _ptr(ws),
        ws.numel(), _stream(dev)))
    if check:
        check_error_word("vt_select_vocab", ws)
    return t2f, f2t, sums


def coverage(sums: torch.Tensor) -> float:
    """kept / total from the sums of select_vocab (synchronises)."""
    kept, total = (int(x) for x in sums.cpu().tolist())
    return float("nan") if total == 0 else kept / total


def gather_rows(W: torch.Tensor, t2f: torch.Tensor,
                out: torch.Tensor | None = None,
                n_invalid: torch.Tensor | None = None) -> torch.Tensor:
    """W_high[i] = W[t2f[i]] for a bf16 [V, d] weight."""
    _cuda(W, "W", torch.bfloat16)
    _cuda(t2f, "t2f", torch.int32)
    V, d = W.shape
    if out is None:
        out = torch.empty(t2f.numel(), d, dtype=torch.bfloat16, device=W.device)
    _cuda(out, "out", torch.bfloat16)
    if n_invalid is not None:
        _cuda(n_invalid, "n_invalid", torch.int64)
    _check("vt_gather_rows", load().vt_gather_rows(
        _ptr(W), V, d, _ptr(t2f), t2f.numel(), _ptr(out), _ptr(n_invalid),
        _stream(W.device)))
    return out


def draft_head(H: torch.Tensor, W_high: torch.Tensor, t2f: torch.Tensor | None,
               k: int, out_ids: torch.Tensor | None = None,
               out_probs: torch.Tensor | None = None,
               out_logits: torch.Tensor | None = None,
               ws: torch.Tensor | None = None, *,
               bias: torch.Tensor | None = None, temperature: float = 1.0,
               sample: bool = False, seed: int = 0, offset: int = 0,
               check: bool = False):
    """One draft step: top-k full-vocabulary ids and softmax probabilities
    over the V_high kept rows for each of the M hidden states in ``H``.
    ``check=True`` synchronises after the call, and raises
    VTError(VT_ERR_TIMEOUT) (clearing the word) if a bounded wait inside the
    head's kernels gave up.

    With options (vt_draft_head_ex): ``bias`` (fp32 [V_high]) is added to
    every logit, probabilities are softmax(logit / temperature), and
    ``sample=True`` draws instead of taking the top-k (k = 1: one draw;
    k > 1: draws without replacement), with the generator keyed by
    ``seed`` and the step counter ``offset``."""
    _cuda(W_high, "W_high", torch.bfloat16)
    if not (isinstance(H, torch.Tensor) and H.is_cuda and H.dtype == torch.bfloat16
            and H.dim() == 2 and H.stride(1) == 1):
        raise TypeError("H must be a CUDA bf16 [M, d] tensor with unit column stride")
    M, d = H.shape
    V_high = W_high.shape[0]
    dev = W_high.device
    if t2f is not None:
        _cuda(t2f, "t2f", torch.int32)
    if out_ids is None:
        out_ids = torch.empty(M, k, dtype=torch.int32, device=dev)
    if out_probs is None:
        out_probs = torch.empty(M, k, dtype=torch.float32, device=dev)
    _cuda(out_ids, "out_ids", torch.int32)
    _cuda(out_probs, "out_probs", torch.float32)
    if out_logits is not None:
        _cuda(out_logits, "out_logits", torch.float32)
    lib = load()
    nbytes = lib.vt_draft_head_workspace_size(M, V_high, k)
    if ws is None:
        ws = _ws.get("head", nbytes, dev, zeroed=True)
    if bias is None and temperature == 1.0 and not sample:
        _check("vt_draft_head", lib.vt_draft_head(
            _ptr(H), M, d, H.stride(0), _ptr(W_high), V_high, _ptr(t2f), k,
            _ptr(out_ids), _ptr(out_probs), _ptr(out_logits), _ptr(ws),
            ws.numel(), _stream(dev)))
        if check:
            check_error_word("vt_draft_head", ws)
        return out_ids, out_probs
    if bias is not None:
        _cuda(bias, "bias", torch.float32)
        if bias.numel() != V_high:
            raise ValueError("bias must hold V_high values")
    opts = HeadOptions(_ptr(bias), float(temperature),
                       VT_HEAD_SAMPLE if sample else VT_HEAD_TOPK,
                       int(seed) & (2**64 - 1), int(offset) & (2**64 - 1))
    _check("vt_draft_head_ex", lib.vt_draft_head_ex(
        _ptr(H), M, d, H.stride(0), _ptr(W_high), V_high, _ptr(t2f), k,
        ctypes.byref(opts), _ptr(out_ids), _ptr(out_probs), _ptr(out_logits),
        _ptr(ws), ws.numel(), _stream(dev)))
    if check:
        check_error_word("vt_draft_head_ex", ws)
    return out_ids, out_probs


def gather_bias(b: torch.Tensor, t2f: torch.Tensor,
                out: torch.Tensor | None = None,
                n_invalid: torch.Tensor | None = None) -> torch.Tensor:
    """b_high = b[t2f]: the kept rows' bias (fp32), for ``bias=`` of
    draft_head."""
    _cuda(b, "b", torch.float32)
    _cuda(t2f, "t2f", torch.int32)
    dev = b.device
    if out is None:
        out = torch.empty(t2f.numel(), dtype=torch.float32, device=dev)
    _cuda(out, "out", torch.float32)
    if n_invalid is not None:
        _cuda(n_invalid, "n_invalid", torch.int64)
    _check("vt_gather_bias", load().vt_gather_bias(
        _ptr(b), b.numel(), _ptr(t2f), t2f.numel(), _ptr(out), _ptr(n_invalid),
        _stream(dev)))
    return out


def draft_head_sets(H: torch.Tensor, set_of_row, W_high_sets, t2f_sets, k: int,
                    bias_sets=None, temperature: float = 1.0,
                    sample: bool = False, seed: int = 0, offset: int = 0,
                    out_ids: torch.Tensor | None = None,
                    out_probs: torch.Tensor | None = None,
                    ws: torch.Tensor | None = None, check: bool = False):
    """One draft step where hidden state m uses kept vocabulary set
    ``set_of_row[m]`` (``W_high_sets[s]``, ``t2f_sets[s]``, optional
    ``bias_sets[s]``); otherwise as draft_head."""
    if not (isinstance(H, torch.Tensor) and H.is_cuda and H.dtype == torch.bfloat16
            and H.dim() == 2 and H.stride(1) == 1):
        raise TypeError("H must be a CUDA bf16 [M, d] tensor with unit column stride")
    M, d = H.shape
    S = len(W_high_sets)
    rows = [int(x) for x in set_of_row]
    if len(rows) != M:
        raise ValueError("set_of_row must name a set for every hidden state")
    for s_, W in enumerate(W_high_sets):
        _cuda(W, f"W_high_sets[{s_}]", torch.bfloat16)
    dev = H.device
    P = ctypes.c_void_p
    W_arr = (P * S)(*[W.data_ptr() for W in W_high_sets])
    V_arr = (ctypes.c_int32 * S)(*[W.shape[0] for W in W_high_sets])
    T_arr = (P * S)(*[None if t is None else _cuda(t, "t2f", torch.int32).data_ptr()
                      for t in (t2f_sets or [None] * S)])
    B_arr = None
    if bias_sets is not None:
        B_arr = (P * S)(*[None if b is None else _cuda(b, "bias", torch.float32).data_ptr()
                          for b in bias_sets])
    sor = (ctypes.c_int32 * M)(*rows)
    if out_ids is None:
        out_ids = torch.empty(M, k, dtype=torch.int32, device=dev)
    if out_probs is None:
        out_probs = torch.empty(M, k, dtype=torch.float32, device=dev)
    lib = load()
    nbytes = lib.vt_draft_head_sets_workspace_size(M, d, k, S, V_arr)
    if ws is None:
        ws = _ws.get("head_sets", nbytes, dev, zeroed=True)
    opts = HeadOptions(None, float(temperature),
                       VT_HEAD_SAMPLE if sample else VT_HEAD_TOPK,
                       int(seed) & (2**64 - 1), int(offset) & (2**64 - 1))
    _check("vt_draft_head_sets", lib.vt_draft_head_sets(
        _ptr(H), M, d, H.stride(0), sor, S, W_arr, V_arr, T_arr, B_arr, k,
        ctypes.byref(opts), _ptr(out_ids), _ptr(out_probs), _ptr(ws),
        ws.numel(), _stream(dev)))
    if check:
        check_error_word("vt_draft_head_sets", ws)
    return out_ids, out_probs


def draft_q(logits: torch.Tensor, f2t: torch.Tensor | None, V: int,
            temperature: float = 1.0, out: torch.Tensor | None = None,
            ws: torch.Tensor | None = None) -> torch.Tensor:
    """Full-vocabulary draft distribution q[M, V] from the head's logits
    [M, V_high] (bias included): softmax(logit / T) at the kept ids (through
    f2t), 0 at dropped ids; ``f2t=None`` is the identity."""
    _cuda(logits, "logits", torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits must be [M, V_high]")
    M, V_high = logits.shape
    dev = logits.device
    if f2t is not None:
        _cuda(f2t, "f2t", torch.int32)
        if f2t.numel() != V:
            raise ValueError("f2t must hold V entries")
    if out is None:
        out = torch.empty(M, V, dtype=torch.float32, device=dev)
    _cuda(out, "out", torch.float32)
    lib = load()
    nbytes = lib.vt_draft_q_workspace_size(M)
    if ws is None:
        ws = _ws.get("draft_q", nbytes, dev, zeroed=True)
    _check("vt_draft_q", lib.vt_draft_q(
        _ptr(logits), M, V_high, _ptr(f2t), V, float(temperature), _ptr(out),
        _ptr(ws), ws.numel(), _stream(dev)))
    return out


def draft_noise(seed: int, offset: int, m: int, full_ids: torch.Tensor,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """The Gumbel noise the sampling head adds to each of ``full_ids``
    (int32, device) for hidden state m at (seed, offset)."""
    _cuda(full_ids, "full_ids", torch.int32)
    dev = full_ids.device
    if out is None:
        out = torch.empty(full_ids.numel(), dtype=torch.float32, device=dev)
    _cuda(out, "out", torch.float32)
    lib = load()
    _check("vt_draft_noise", lib.vt_draft_noise(
        int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), m, _ptr(full_ids),
        full_ids.numel(), _ptr(out), _stream(dev)))
    return out


def draft_head_host(H_host: torch.Tensor, W_high: torch.Tensor,
                    t2f: torch.Tensor | None, k: int,
                    H_dev: torch.Tensor | None = None,
                    ids_host: torch.Tensor | None = None,
                    probs_host: torch.Tensor | None = None):
    """End-to-end call from host memory: copies H (pinned host) to the
    device, runs draft_head, copies ids/probs back, and synchronises."""
    dev = W_high.device
    if H_dev is None:
        H_dev = torch.empty(H_host.shape, dtype=torch.bfloat16, device=dev)
    H_dev.copy_(H_host, non_blocking=True)
    ids, probs = draft_head(H_dev, W_high, t2f, k)
    if ids_host is None:
        ids_host = torch.empty(ids.shape, dtype=torch.int32, pin_memory=True)
    if probs_host is None:
        probs_host = torch.empty(probs.shape, dtype=torch.float32, pin_memory=True)
    ids_host.copy_(ids, non_blocking=True)
    probs_host.copy_(probs, non_blocking=True)
    torch.cuda.current_stream(dev).synchronize()
    return ids_host, probs_host


class HostDraftHead:
    """Draft steps from host memory through the library's host step
    (vt_host_step_*): each call copies the hidden states into the handle's
    pinned staging buffer, launches one CUDA graph (copy in, then the head,
    whose kernel writes ids and probabilities into pinned host memory, then
    a kernel that publishes the step's sequence number there), waits for
    that number, and returns host tensors (ids [M, k] int32, probs [M, k]
    float32) that the next call overwrites.  ``W_high``, ``t2f``, ``k``, M and the options (bias,
    temperature) are fixed; drawing is not offered (a replayed graph repeats
    its step counter).  Write ``head.H_host`` in place and call ``head()``
    to skip the host copy."""

    def __init__(self, W_high: torch.Tensor, t2f: torch.Tensor | None, k: int,
                 M: int, bias: torch.Tensor | None = None,
                 temperature: float = 1.0):
        _cuda(W_high, "W_high", torch.bfloat16)
        if t2f is not None:
            _cuda(t2f, "t2f", torch.int32)
        if bias is not None:
            _cuda(bias, "bias", torch.float32)
        V_high, d = W_high.shape
        self.M, self.k = M, k
        self._keep = (W_high, t2f, bias)  # the graph reads these
        lib = load()
        opts = HeadOptions(_ptr(bias), float(temperature), VT_HEAD_TOPK, 0, 0)
        h = ctypes.c_void_p()
        with torch.cuda.device(W_high.device):
            _check("vt_host_step_create", lib.vt_host_step_create(
                _ptr(W_high), V_high, d, _ptr(t2f), M, k, ctypes.byref(opts),
                ctypes.byref(h)))
        self._h = h
        staging = lib.vt_host_step_staging(h)
        buf = (ctypes.c_uint16 * (M * d)).from_address(staging)
        self.H_host = torch.frombuffer(buf, dtype=torch.int16).view(
            torch.bfloat16).view(M, d)
        self.ids = torch.empty(M, k, dtype=torch.int32)
        self.probs = torch.empty(M, k, dtype=torch.float32)
        self._lib = lib
        # per-step call: the entry point and the output pointers, looked up once
        self._run = lib.vt_host_step_run
        self._shape = (M, d)
        self._staging = staging
        self._out = (self.ids.data_ptr(), self.probs.data_ptr())

    @property
    def error_word(self) -> int:
        """Device address of the handle's error word (uint32): a step whose
        head finds it set raises VTError(VT_ERR_TIMEOUT) and clears it."""
        return self._lib.vt_host_step_error_word(self._h)

    def __call__(self, H_host: torch.Tensor | None = None):
        if H_host is None:
            src = self._staging
        else:
            if (H_host.dtype != torch.bfloat16 or H_host.is_cuda
                    or tuple(H_host.shape) != self._shape):
                raise TypeError(f"H_host must be a host bf16 tensor of shape {self._shape}")
            if not H_host.is_contiguous():
                H_host = H_host.contiguous()  # (kept alive through the call)
            src = H_host.data_ptr()
        status = self._run(self._h, src, *self._out)
        if status != VT_OK:
            _check("vt_host_step_run", status)
        return self.ids, self.probs

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.vt_host_step_destroy(h)
            self._h = None


def build_vocab(tokens: torch.Tensor, V: int, V_high: int,
                W: torch.Tensor | None = None, b: torch.Tensor | None = None):
    """The offline build in one call: histogram, selection, maps and (if
    ``W`` / ``b`` are given) the gathered W_high / b_high.  Returns a dict of
    device tensors."""
    counts, n_invalid = count_tokens(tokens, V)
    t2f, f2t, sums = select_vocab(counts, V_high)
    out = dict(counts=counts, n_invalid=n_invalid, t2f=t2f, f2t=f2t, sums=sums)
    if W is not None:
        out["W_high"] = gather_rows(W, t2f)
    if b is not None:
        out["b_high"] = gather_bias(b, t2f)
    return out


_VOCAB_FORMAT = 1


def save_vocab(path: str, vocab: dict) -> None:
    """Writes the offline build's result (the output of ``build_vocab``:
    counts, t2f, f2t, sums and n_invalid; not W_high, which is rebuilt from
    the model's weights with ``gather_rows``) to a ``.npz`` file, so a
    serving process can load the kept vocabulary instead of recounting the
    corpus."""
    import numpy as np
    arrays = {"format": np.array([_VOCAB_FORMAT], dtype=np.int64)}
    for key in ("counts", "t2f", "f2t", "sums", "n_invalid"):
        t = vocab[key].detach().cpu()
        if t.dtype == torch.uint32:
            t = t.view(torch.int32)  # stored as raw 32-bit words
        arrays[key] = t.numpy()
    np.savez(path, **arrays)


def load_vocab(path: str, device: torch.device | str = "cuda") -> dict:
    """Reads a file written by ``save_vocab``; returns the same tensors
    (counts uint32[V], t2f int32[V_high], f2t int32[V], sums int64[2],
    n_invalid int64[1]) on ``device``, checked for consistency: t2f and f2t
    are inverse maps over the kept ids and V_high <= V."""
    import numpy as np
    with np.load(path) as z:
        if int(z["format"][0]) != _VOCAB_FORMAT:
            raise ValueError(f"{path}: unknown vocabulary file format")
        arr = {k: z[k] for k in ("counts", "t2f", "f2t", "sums", "n_invalid")}
    t2f, f2t = arr["t2f"], arr["f2t"]
    V, V_high = f2t.size, t2f.size
    if (arr["counts"].size != V or V_high > V or t2f.min(initial=0) < 0
            or t2f.max(initial=0) >= V
            or not np.array_equal(f2t[t2f], np.arange(V_high))
            or int((f2t >= 0).sum()) != V_high):
        raise ValueError(f"{path}: maps are not consistent")
    out = {k: torch.from_numpy(v).to(device) for k, v in arr.items()}
    out["counts"] = out["counts"].view(torch.uint32)
    return out
