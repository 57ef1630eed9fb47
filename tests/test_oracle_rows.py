"""The GPU tests run the oracle over many rows in threads (gpu_util.
oracle_head); on the CPU, check that the joined result is exactly one call
over all rows, for top-k and for draws (whose noise index counts the rows
of the whole call)."""
import numpy as np

import oracle
import synth
from gpu_util import oracle_head


def test_threaded_rows_equal_one_call(oracle_lib):
    M, d, V_high, k = 37, 64, 900, 6
    Hh = synth.bf16_bits(synth.normal_bf16((M, d), 1.0, seed=51))
    Wh = synth.bf16_bits(synth.normal_bf16((V_high, d), 0.1, seed=52))
    t2f = synth.rank_permutation(2000, 53)[:V_high].numpy()
    ref, full = oracle_head(Hh, Wh, t2f, k)
    one = oracle.draft_head(Hh, Wh, t2f, k)
    for key in one:
        assert np.array_equal(ref[key], one[key]), key
    assert np.array_equal(full, oracle.head_logits(Hh, Wh))
    opts = dict(sample=True, seed=9, offset=4, temperature=0.9)
    ref, _ = oracle_head(Hh, Wh, t2f, k, logits=False, m_base=3, **opts)
    one = oracle.draft_head_ex(Hh, Wh, t2f, k, m_base=3, **opts)
    for key in one:
        assert np.array_equal(ref[key], one[key]), key
