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

# Mistakes in the head's options (bias, temperature, sampling); these are
# run against the options pins.
OPTION_MUTANTS = {
    "gumbel_sign": ("return -std::log(-std::log(u));",
                    "return std::log(-std::log(u));"),
    "exponential_not_gumbel": ("return -std::log(-std::log(u));",
                               "return -std::log(u);"),
    "uniform_wrong_scale": ("+ 0.5) / 8388608.0;", "+ 0.5) / 16777216.0;"),
    "temperature_multiplies": ("s[i] = logits[i] / temperature;",
                               "s[i] = logits[i] * temperature;"),
    "bias_dropped": ("logits[i] += bias_high ? static_cast<double>(bias_high[i]) : 0.0;",
                     "logits[i] += 0.0;"),
    "philox_no_key_bump": ("k[0] += kWeyl0;", "k[0] += 0u;"),
    "philox_swapped_halves": ("c[1] = lo1;", "c[1] = lo0;"),
    "noise_by_trimmed_index": ("gumbel_noise(seed, offset, m_base + m, full_id(i))",
                               "gumbel_noise(seed, offset, m_base + m, i)"),
    "noise_row_ignores_m_base": ("gumbel_noise(seed, offset, m_base + m, full_id(i))",
                                 "gumbel_noise(seed, offset, m, full_id(i))"),
    "noise_ignores_row": ("static_cast<uint32_t>(full_id), static_cast<uint32_t>(m),",
                          "static_cast<uint32_t>(full_id), 0u,"),
    "noise_ignores_offset_high": ("static_cast<uint32_t>(offset >> 32)};",
                                  "0u};"),
    "bias_gather_wrong_index": ("b_high[i] = b[src];", "b_high[i] = b[i];"),
    "q_placed_by_position": ("      const int32_t f = t2f ? t2f[i] : i;\n      if (f < 0 || f >= V) return 2;",
                             "      const int32_t f = i;\n      if (f < 0 || f >= V) return 2;"),
    "q_without_temperature": ("             temperature;\n    double mx = s[0];",
                              "             1.0;\n    double mx = s[0];"),
    "sample_prob_of_score": ("if (probs) probs[o] = std::exp(s[i] - mx) / sumexp;\n      if (scores)",
                             "if (probs) probs[o] = std::exp(key[i] - mx) / sumexp;\n      if (scores)"),
}


ALL = {**{n: (m, "test_oracle_pins.py") for n, m in MUTANTS.items()},
       **{n: (m, "test_oracle_pins_options.py")
          for n, m in OPTION_MUTANTS.items()}}


@pytest.mark.parametrize("name", sorted(ALL))
def test_pins_catch_mutant(name, tmp_path):
    (old, new), pins = ALL[name]
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
                        os.path.join(ROOT, "tests", pins)],
                       env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"no pin caught mutant {name}:\n{r.stdout[-2000:]}"
