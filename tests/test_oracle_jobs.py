"""The per-request oracle jobs of the full-size parity tests (CPU): the process pool returns, for every
request, exactly what the oracle computes on the whole batch."""
import numpy as np

import oracle
from synth import cpu as gen
from synth import recipe
from tests import oracle_jobs


def test_pool_matches_the_oracle_on_the_whole_batch():
    w = recipe.small(lengths=(700, 0, 90, 333), Hq=4, Hkv=2, dk=64, hdim=64, G=32, n=64, salt=5)
    host = gen.materialize(w, with_hidden=False)
    Q = gen.bf16_bits_to_f32(host["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(host["K"]).astype(np.float64)
    ref = oracle.block_scores(Q, K, host["cu_seqlens"], w.G, w.n)
    cb = oracle.cu_blocks_of(host["cu_seqlens"], w.G)
    got = oracle_jobs.all_block_scores(w, host["u"], host["hot_tok"])
    assert sorted(got) == list(range(w.R))
    for r in range(w.R):
        assert np.array_equal(got[r], ref[cb[r]:cb[r + 1]])
