"""Seeded synthetic inputs shared by the CUDA path and the oracle.

This module holds input generation only: none of the method's arithmetic
(no counting, selection, projection, softmax or top-k) lives here.  Both
sides of every parity test consume the very same bytes produced here.

Recipe (stands in for the corpora and model weights the pages use, which are
not available):
  * token streams: i.i.d. Zipf(s) ranks over 1..V drawn by inverse CDF
    (fp64 uniform from a seeded torch generator, ``searchsorted`` into an
    fp64 CDF table), then mapped rank -> id through a seeded random
    permutation, so frequent ids are scattered over the id range;
  * weights W ~ N(0, 0.02) and hidden states H ~ N(0, 1), drawn in fp32 from
    a seeded torch generator and rounded once to bf16 (round to nearest even).
The generator runs on CPU or CUDA; a given call is reproducible on its own
device.  Tests that compare against the oracle draw once and hand the same
tensor (or its host copy) to both sides.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


def zipf_cdf(V: int, s: float) -> np.ndarray:
    """fp64 CDF of Zipf(s) over ranks 1..V (last entry forced to 1.0)."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    w = ranks ** (-s)
    cdf = np.cumsum(w) / w.sum()
    cdf[-1] = 1.0
    return cdf


def rank_permutation(V: int, seed: int) -> torch.Tensor:
    """Seeded permutation rank -> token id (int32, on CPU)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randperm(V, generator=g).to(torch.int32)


def zipf_tokens(n: int, V: int, s: float = 1.1, seed: int = 0,
                device: str | torch.device = "cpu",
                chunk: int = 1 << 26) -> torch.Tensor:
    """``n`` int32 token ids, Zipf(s) over a seeded rank->id permutation."""
    device = torch.device(device)
    cdf = torch.from_numpy(zipf_cdf(V, s)).to(device)
    perm = rank_permutation(V, seed ^ 0x5EED).to(device)
    g = torch.Generator(device=device).manual_seed(seed)
    out = torch.empty(n, dtype=torch.int32, device=device)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        u = torch.rand(hi - lo, dtype=torch.float64, generator=g,
                       device=device)
        r = torch.searchsorted(cdf, u, right=True).clamp_(max=V - 1)
        out[lo:hi] = perm[r]
        del u, r
    return out


def normal_bf16(shape, std: float, seed: int,
                device: str | torch.device = "cpu") -> torch.Tensor:
    """bf16 tensor ~ N(0, std^2): fp32 draw from a seeded generator, RNE."""
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def expected_rank_ids(V: int, V_high: int, seed: int) -> torch.Tensor:
    """The V_high most likely ids of the seeded Zipf stream, rank order.

    This is the expected frequency ranking of ``zipf_tokens(..., seed)``
    (the permutation's first V_high entries).  It stands in for a measured
    ranking where a workload only needs *a* frequency-ranked row set.
    """
    return rank_permutation(V, seed ^ 0x5EED)[:V_high].clone()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 view of a bf16 tensor's bit patterns (for the oracle)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(
        np.uint16)


@dataclasses.dataclass(frozen=True)
class HeadShape:
    name: str
    d: int
    V: int
    V_high: int
    M: int
    k: int
    seed: int


@dataclasses.dataclass(frozen=True)
class BuildShape:
    name: str
    n_tokens: int
    V: int
    V_high: int
    d: int
    s: float
    seed: int


# The workloads (sizes, distributions) of the pages' evaluation, at the
# shapes of the drafter heads they name.  Seeds are fixed per workload.
TINY_BUILD = BuildShape("tiny d=256 V=4096 V_high=1024 n=1e6", 1_000_000,
                        4096, 1024, 256, 1.1, 1001)
TINY_HEAD = HeadShape("tiny d=256 V_high=1024 M=1 k=8", 256, 4096, 1024, 1,
                      8, 1001)
LLAMA8B_HEAD = HeadShape("llama3-8b head d=4096 V=128256 V_high=32768 M=1 k=10",
                         4096, 128256, 32768, 1, 10, 1002)
TREE_HEAD = HeadShape("eagle2 tree d=4096 V=128256 M=60 k=10", 4096, 128256,
                      32768, 60, 10, 1003)
TREE_V_HIGH_SWEEP = (8192, 16384, 32768, 65536, 128256)
QWEN7B_HEAD = HeadShape("qwen2-7b head d=3584 V=152064 V_high=32768", 3584,
                        152064, 32768, 1, 10, 1004)
LLAMA1B_HEAD = HeadShape("llama3.2-1b head d=2048 V=128256 V_high=32768", 2048,
                         128256, 32768, 1, 10, 1004)
M_SWEEP = (1, 4, 16, 64)
SCALE_BUILD = BuildShape("vocab build n=1e9 V=128256 V_high=32768 d=4096",
                         1_000_000_000, 128256, 32768, 4096, 1.1, 1005)
