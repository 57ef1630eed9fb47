"""The committed ncu summaries, without a GPU: the M = 1 head's summary was
taken on the current kernel sources (so the bench reports its DRAM traffic
rather than null), every summary gives the command that made it with
`--clock-control none`, and nothing but short text summaries is kept."""
import importlib.util
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_head_traffic_summary_matches_current_sources():
    bench = _bench()
    traffic = bench.committed_traffic()
    assert traffic is not None, (
        "profiles/head_gemv_llama8b_m1.md was taken on other kernel sources: "
        "re-capture it and record the new kernel_source_sha256")
    # DRAM bytes of one launch sit just above the algorithmic bytes
    assert 268_443_728 <= traffic <= 1.05 * 268_443_728


def test_every_summary_names_its_command():
    names = sorted(os.listdir(PROFILES))
    assert names, "no profiles committed"
    for name in names:
        assert name.endswith((".md", ".txt")), f"{name}: only text summaries belong here"
        text = open(os.path.join(PROFILES, name)).read()
        assert len(text) < 20_000, f"{name}: a summary, not a raw report"
        cmds = re.findall(r"^ncu .*$", text, flags=re.M)
        assert cmds, f"{name}: no ncu command line"
        for c in cmds:
            assert "--clock-control none" in c, f"{name}: {c}"
