"""Planted mistakes: each mutant is the oracle source with one plausible
error (a dropped term, a wrong sign, a wrong index, a flipped tie rule).
Each is compiled on the CPU into a temporary library and the pin suite is
run against it; every mutant must make at least one pin fail.  The mistakes
live only in temporary copies, never in the committed oracle."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = {
    "count_twice": ("token_counts[id] += 1;", "token_counts[id] += 2;"),
    "valid_off_by_one": ("id >= V", "id > V"),
    "tie_higher_id": ("return a.id < b.id;", "return a.id > b.id;"),
    "ascending_count": ("return a.count > b.count;", "return a.count < b.count;"),
    "f2t_shifted": ("f2t[items[i].id] = i;", "f2t[items[i].id] = i + 1;"),
    "coverage_wrong_total": ("total_count += counts[id];",
                             "total_count += counts[id] + (id == 0);"),
    "gather_wrong_row": ("W + src * d", "W + static_cast<int64_t>(i) * d"),
    "dot_drops_last_term": ("for (int32_t j = 0; j < d; ++j)\n",
                            "for (int32_t j = 0; j < d - 1; ++j)\n"),
    "dot_transposed": ("bf16_to_double(h[j]) * bf16_to_double(w[j])",
                       "bf16_to_double(h[j]) * bf16_to_double(W_high[static_cast<int64_t>(j % V_high) * d + i % d])"),
    "softmax_sign": ("sumexp += std::exp(logits[i] - mx);",
                     "sumexp += std::exp(mx - logits[i]);"),
    "softmax_no_max": ("sumexp += std::exp(logits[i] - mx);",
                       "sumexp += std::exp(logits[i]) / std::exp(mx);"),
    "topk_tie_trimmed_index": ("return full_id(a) < full_id(b);",
                               "return a < b;"),
    "no_remap": ("if (ids) ids[o] = full_id(i);", "if (ids) ids[o] = i;"),
    "prob_denominator": ("std::exp(logits[i] - mx) / sumexp;",
                         "std::exp(logits[i] - mx) / (sumexp + 1e-9);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    cpp = tmp_path / "mutant.cpp"
    cpp.write_text(mutated)
    lib = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", str(cpp),
                    "-o", str(lib)], check=True)
    env = dict(os.environ, FRD_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p",
                        "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"no pin caught mutant {name}:\n{r.stdout[-2000:]}"
