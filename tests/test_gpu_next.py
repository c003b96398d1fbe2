"""Widening beyond the single drop step (GPU): the tensor-parallel score split of Eq. 15 emulated on one
GPU, and the decode-side metadata of two drop events in a chain (Eqs. 16-17 with per-layer tables)."""
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


def _scores(w, host):
    d = sgpu.to_device(host)
    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, 0, G=w.G, n=w.n, A=w.A, p=w.p)
    step.score(d["Q"], d["K"])
    torch.cuda.synchronize()
    step.check()
    return step


def test_head_split_eq15_sum_gives_the_unsplit_decision():
    """UniPrefill section 3.5, Eq. 15: each tensor-parallel rank scores its own query heads (with their KV
    heads) and the ranks' block scores are summed before top-p.  Two ranks of equal head counts: each rank's
    scores are the mean over its heads, so the sum is twice the unsplit mean, and top-p on the sum keeps the
    unsplit set (up to blocks within the selection tolerance of the threshold)."""
    w = recipe.small(lengths=(1500, 700, 2100, 90), Hq=8, Hkv=4, dk=128, hdim=64, G=64, n=128, p=0.95, salt=151)
    host = gen.materialize(w, with_hidden=False)
    full = _scores(w, host)
    b_full = full.block_scores.cpu().numpy().astype(np.float64)[:full.nb_cap]
    ranks = 2
    hq, hkv = w.Hq // ranks, w.Hkv // ranks
    b_sum = np.zeros_like(b_full)
    for t in range(ranks):
        ht = dict(host)
        ht["Q"] = np.ascontiguousarray(host["Q"][:, t * hq:(t + 1) * hq])
        ht["K"] = np.ascontiguousarray(host["K"][:, t * hkv:(t + 1) * hkv])
        st = _scores(w.replace(Hq=hq, Hkv=hkv), ht)
        b_sum += st.block_scores.cpu().numpy().astype(np.float64)[:full.nb_cap]
    cb = oracle.cu_blocks_of(host["cu_seqlens"], w.G)
    nbt = int(cb[-1])
    parity.check_block_scores(b_sum[:nbt] / ranks, b_full[:nbt], rtol=1e-5)
    # top-p on the summed scores (the selection kernel, on device) against the unsplit scores' decision
    full.block_scores[:nbt] = torch.from_numpy(b_sum[:nbt].astype(np.float32)).cuda()
    full.select()
    torch.cuda.synchronize()
    full.check()
    parity.check_selection(full.block_keep.cpu().numpy()[:nbt], full.token_keep.cpu().numpy(), b_full[:nbt],
                           host["cu_seqlens"], w.G, w.n, w.A, w.p)


def test_two_drop_events_keep_the_decode_metadata_consistent():
    """Two drop steps in one 8-layer stack, at layers 2 and 5, the second on the stream the first compacted
    (Eqs. 7-8: the sublayers in between run on the kept tokens; their Q/K rows stand in for the recomputed
    ones).  The recorded history gives Eq. 17's seqused for every layer with decode tokens appended (kv_len >
    orig_len), the twice-gathered positions and slots are the originals of the doubly kept tokens, and Eq. 16
    with a different block table per layer reproduces each layer's slots of the compacted stream."""
    L, drops = 8, (2, 5)
    w = recipe.small(lengths=(1800, 130, 2500, 600), Hq=8, Hkv=2, dk=128, hdim=64, G=64, n=128, A=128, p=0.9,
                     hot=("frac", 0.2), salt=171)
    host = gen.materialize(w, with_hidden=False)
    cu0 = host["cu_seqlens"]
    R = w.R
    d = sgpu.to_device(host)
    # drop 1 at layer 2 on the full stream
    a = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, 0, G=w.G, n=w.n, A=w.A, p=w.p, L=L, layer=drops[0])
    a.score(d["Q"], d["K"])
    a.select()
    a.compact(None, d["positions"], d["slots"])
    torch.cuda.synchronize()
    a.check()
    tka = a.token_keep.cpu().numpy()
    ref_a = oracle.compact(tka, cu0, None, host["positions"], host["slots"])
    Ta = ref_a["num_actual_tokens"]
    ka = a.kept_index.cpu().numpy()[:Ta]
    assert np.array_equal(ka, ref_a["kept_index"])
    # drop 2 at layer 5 on the compacted stream, with the history of drop 1 carried in its buffers
    cua = a.new_cu.cpu().numpy()
    qa = d["Q"][torch.from_numpy(ka.astype(np.int64)).cuda()].contiguous()
    kb = d["K"][torch.from_numpy(ka.astype(np.int64)).cuda()].contiguous()
    b = up.DropStep(a.new_cu, Ta, w.Hq, w.Hkv, w.dk, 0, G=w.G, n=w.n, A=w.A, p=w.p, L=L, layer=drops[1])
    b.kept_len.copy_(a.kept_len)
    b.drop_layer.copy_(a.drop_layer)
    b.score(qa, kb)
    b.select()
    b.compact(None, a.out_positions[:Ta], a.out_slots[:Ta])
    torch.cuda.synchronize()
    b.check()
    tkb = b.token_keep.cpu().numpy()
    ref_b = oracle.compact(tkb, cua, None, ref_a["positions"], ref_a["slots"])
    Tb = ref_b["num_actual_tokens"]
    kbi = b.kept_index.cpu().numpy()[:Tb]
    assert np.array_equal(kbi, ref_b["kept_index"])
    cub = b.new_cu.cpu().numpy()
    assert np.array_equal(cub, ref_b["new_cu_seqlens"])
    # composition of the two gathers: the original positions and slots of the doubly kept tokens
    src = ka[kbi]
    assert np.array_equal(b.out_positions.cpu().numpy()[:Tb], host["positions"][src])
    assert np.array_equal(b.out_slots.cpu().numpy()[:Tb], host["slots"][src])
    # the drop history and Eq. 17 for every layer, with decode tokens appended
    kept_ref = np.zeros((L, R), dtype=np.int32)
    kept_ref[drops[0]] = ref_a["seq_lens"]
    kept_ref[drops[1]] = ref_b["seq_lens"]
    drop_ref = np.zeros(L, dtype=np.uint8)
    drop_ref[list(drops)] = 1
    got_kept = b.kept_len.cpu().numpy()
    assert np.array_equal(got_kept[list(drops)], kept_ref[list(drops)])
    assert np.array_equal(b.drop_layer.cpu().numpy(), drop_ref)
    orig = np.diff(cu0).astype(np.int32)
    kv = (orig + np.array([3, 0, 7, 1], dtype=np.int32)).astype(np.int32)
    orig_t, kv_t = torch.from_numpy(orig).cuda(), torch.from_numpy(kv).cuda()
    for layer in range(L):
        got = b.seqused(orig_t, kv_t, layer).cpu().numpy()
        assert np.array_equal(got, oracle.seqused(kept_ref, drop_ref, layer, orig, kv)), layer
    # Eq. 16 per layer after the second drop, a different block table each (B = 16)
    B = 16
    mb = int(max(host["positions"].max() // B + 1, 1))
    rng = np.random.default_rng(16)
    pos_b = b.out_positions[:Tb].contiguous()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for layer in range(drops[1] + 1, L):
        table = rng.permutation(R * mb).reshape(R, mb).astype(np.int32)
        slots = torch.zeros(max(1, Tb), dtype=torch.int64, device="cuda")
        up.up_slot_mapping(pos_b, b.new_cu, torch.from_numpy(table).cuda(), B, slots, status)
        assert up.up_read_status(status) == 0
        assert np.array_equal(slots.cpu().numpy()[:Tb], oracle.slot_mapping(host["positions"][src], cub, table, B))
