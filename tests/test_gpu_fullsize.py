"""Full-size parity: the five workloads at their real sizes, generated on the device and run through
the same DropStep calls that bench.py times; the oracle checks sampled requests (block scores and
the kept-block set, with the stated tolerances) and sampled hidden rows, and the whole compaction
index and metadata (bit-exact given the GPU's mask)."""
import numpy as np
import pytest
import torch

import long_context_prefill_varlen_gb300 as up
import oracle
from synth import cpu as gen
from synth import gpu as sgpu
from synth import recipe
from tests import parity

pytestmark = pytest.mark.gpu

# requests whose scores the oracle recomputes, per workload
SAMPLED = {2: [0], 3: "shortest+median", 4: [1], 5: [0, 37]}


def _sampled_requests(w, spec):
    if spec == "shortest+median":
        order = np.argsort(w.lengths)
        return [int(order[0]), int(order[len(order) // 2])]
    return list(spec)


def _oracle_request(w, r, u, hot_tok):
    cu = w.cu_seqlens()
    a, b = cu[r], cu[r + 1]
    N = b - a
    ne = min(w.n, N)
    Q = np.zeros((N, w.Hq, w.dk))
    Q[N - ne:] = gen.bf16_bits_to_f32(gen.gen_q(w, b - ne, b))
    K = gen.bf16_bits_to_f32(gen.gen_k(w, a, b, u, hot_tok)).astype(np.float64)
    return oracle.block_scores(Q, K, [0, N], w.G, w.n)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_fullsize_workload(cfg):
    w = recipe.workload(cfg)
    u = gen.mean_query_dirs(w)
    hot_tok = gen.hot_token_mask(w)
    d = sgpu.build_device(w, u=u, hot_tok=hot_tok)
    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n, A=w.A, p=w.p, L=2, layer=0)
    residual = d["hidden"].clone()
    step.run(d["Q"], d["K"], d["hidden"], d["positions"], d["slots"], residual=residual)
    torch.cuda.synchronize()
    step.check()

    cu = np.asarray(w.cu_seqlens())
    cb = oracle.cu_blocks_of(cu, w.G)
    bs = step.block_scores.cpu().numpy()
    bk = step.block_keep.cpu().numpy()
    tk = step.token_keep.cpu().numpy()
    # the mass invariant holds for every request at any size: sum_g b_g = 1/G
    for r in range(w.R):
        assert abs(bs[cb[r]:cb[r + 1]].astype(np.float64).sum() * w.G - 1.0) < 1e-3
    boundary = 0
    for r in _sampled_requests(w, SAMPLED[cfg]):
        ref = _oracle_request(w, r, u, hot_tok)
        parity.check_block_scores(bs[cb[r]:cb[r + 1]], ref)
        boundary += parity.check_selection(bk[cb[r]:cb[r + 1]], tk[cu[r]:cu[r + 1]], ref, [0, cu[r + 1] - cu[r]],
                                           w.G, w.n, w.A, w.p)
    # compaction index and metadata: whole arrays, bit-exact given the GPU mask
    ref = oracle.compact(tk, cu)
    Tp = ref["num_actual_tokens"]
    assert int(step.num_actual.item()) == Tp
    ki = step.kept_index.cpu().numpy()[:Tp]
    assert np.array_equal(ki, ref["kept_index"])
    assert np.array_equal(step.new_cu.cpu().numpy(), ref["new_cu_seqlens"])
    assert np.array_equal(step.kept_len.cpu().numpy()[0], ref["seq_lens"])
    assert np.array_equal(step.out_positions.cpu().numpy()[:Tp], gen.gen_positions(w)[ki])
    assert np.array_equal(step.out_slots.cpu().numpy()[:Tp], gen.gen_slots(w)[ki])
    # sampled compacted rows against the generator's own rows
    rng = np.random.default_rng(cfg)
    for k in rng.choice(Tp, size=min(Tp, 64), replace=False):
        src = int(ki[k])
        row = step.out_hidden[k].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(row, gen.gen_hidden(w, src, src + 1)[0]), (k, src)
    # Eq. 8 with identity sublayers gives back the block input, byte for byte
    assert torch.equal(residual.view(torch.int16), d["hidden"].view(torch.int16))
    print(f"config {cfg}: T={w.T} T'={Tp} rho={Tp / w.T:.4f} boundary blocks={boundary}")
