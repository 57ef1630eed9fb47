"""The vocabulary file (save_vocab / load_vocab): the offline build's counts,
maps and sums round-trip bit for bit, and a file whose maps disagree is
refused.  Host only (tensors on the CPU)."""
import numpy as np
import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
import oracle


def vocab_from_oracle(V=5000, V_high=777, seed=3):
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 1000, V).astype(np.uint64)
    sel = oracle.select_vocab(counts, V_high)
    return dict(
        counts=torch.from_numpy(counts.astype(np.uint32).view(np.int32)).view(torch.uint32),
        t2f=torch.from_numpy(sel["t2f"]), f2t=torch.from_numpy(sel["f2t"]),
        sums=torch.tensor([int(sel["kept"]), int(sel["total"])], dtype=torch.int64),
        n_invalid=torch.zeros(1, dtype=torch.int64))


def test_round_trip(tmp_path, oracle_lib):
    v = vocab_from_oracle()
    p = str(tmp_path / "vocab.npz")
    vt.save_vocab(p, v)
    w = vt.load_vocab(p, device="cpu")
    for key in v:
        assert w[key].dtype == v[key].dtype, key
        assert torch.equal(w[key].view(torch.int32) if w[key].dtype == torch.uint32 else w[key],
                           v[key].view(torch.int32) if v[key].dtype == torch.uint32 else v[key]), key


def test_inconsistent_maps_are_refused(tmp_path, oracle_lib):
    v = vocab_from_oracle()
    v["f2t"] = v["f2t"].clone()
    kept = int(v["t2f"][5])
    v["f2t"][kept] = 6  # no longer the inverse of t2f
    p = str(tmp_path / "bad.npz")
    vt.save_vocab(p, v)
    with pytest.raises(ValueError):
        vt.load_vocab(p, device="cpu")
