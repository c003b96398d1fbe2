"""The drop step inside a random-weight decoder stack (GPU): UniPrefill section 3.4, Eqs. 7-8.

A 4-layer LLaMA-shaped stack (library layers: cuBLAS GEMMs, PyTorch's varlen flash attention) with drops
at layers 1 and 2.  Each drop's block scores and keep mask are checked against the oracle on the rotated
Q and K the layer produced, and its compaction bit-exactly against the oracle's; the stack's output is
checked against a float64 CPU recomputation that applies the same masks; the rows each drop removed
leave the stack bit-identical to the stream that entered the drop layer (Eq. 8)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_prefill_varlen_gb300 import layerstack as ls
from synth import cpu as gen
from synth import gpu as sgpu
from synth import recipe
from tests import parity
from tests import stack_ref

pytestmark = pytest.mark.gpu

GEOM = ls.StackGeometry(d=256, Hq=4, Hkv=2, dk=64, ffn=512)
LENGTHS = (1500, 700, 0, 2100, 90)
G, n, A = 64, 128, 128
REL_FRO = 2e-2          # bf16 activations through 4 layers against float64
REL_ROW = 6e-2


def _setup():
    w = recipe.small(lengths=LENGTHS, Hq=GEOM.Hq, Hkv=GEOM.Hkv, dk=GEOM.dk, hdim=GEOM.d, G=G, n=n, A=A, salt=257)
    host = gen.materialize(w)
    d = sgpu.to_device(host)
    stack = ls.RandomLlamaStack(4, GEOM, seed=11, device="cuda", init_device="cpu")
    return w, host, d, stack


def _rel_errors(got, ref):
    got = got.double().cpu()
    fro = float(torch.linalg.norm(got - ref) / torch.linalg.norm(ref))
    rows = torch.linalg.norm(got - ref, dim=1) / torch.linalg.norm(ref, dim=1).clamp_min(1e-30)
    return fro, float(rows.max()) if rows.numel() else 0.0


def _hidden_f64(host):
    return torch.from_numpy(gen.bf16_bits_to_f32(host["hidden"]).astype(np.float64))


def test_stack_without_a_drop_matches_the_float64_recomputation():
    w, host, d, stack = _setup()
    out, info = stack.forward(d["hidden"], d["positions"], d["cu_seqlens"], max(LENGTHS))
    torch.cuda.synchronize()
    assert info == []
    ref = stack_ref.forward(stack, _hidden_f64(host), host["positions"], LENGTHS)
    fro, row = _rel_errors(out, ref)
    assert fro < REL_FRO and row < REL_ROW, (fro, row)


def test_two_drops_in_the_stack():
    w, host, d, stack = _setup()
    drops = [(1, 0.8), (2, 0.9)]
    out, info = stack.forward(d["hidden"], d["positions"], d["cu_seqlens"], max(LENGTHS), drops=drops, G=G, n=n,
                              A=A, keep_scored=True)
    torch.cuda.synchronize()
    assert [i["layer"] for i in info] == [1, 2]
    cu = host["cu_seqlens"]
    masks = []
    for i, (layer, p) in zip(info, drops):
        st = i["step"]
        q, k, x, pos = i["scored"]
        Q = q.float().cpu().numpy().astype(np.float64)
        K = k.float().cpu().numpy().astype(np.float64)
        ref_scores = oracle.block_scores(Q, K, cu, G, n)
        got = parity.step_to_numpy(st)
        nbt = len(ref_scores)
        parity.check_block_scores(got["block_scores"][:nbt], ref_scores)
        parity.check_selection(got["block_keep"][:nbt], got["token_keep"], ref_scores, cu, G, n, A, p)
        xb = x.cpu().view(torch.int16).numpy().view(np.uint16)
        Tp = parity.check_compaction(got, got["token_keep"], cu, hidden=xb, positions=pos.cpu().numpy(),
                                     L=stack.L, layer=layer)
        assert Tp == i["kept_tokens"] < len(got["token_keep"])          # the drop removed something
        masks.append((layer, got["token_keep"].astype(bool)))
        cu = got["new_cu"]
    # the whole stack against the float64 recomputation with the same masks
    ref = stack_ref.forward(stack, _hidden_f64(host), host["positions"], LENGTHS, masks)
    fro, row = _rel_errors(out, ref)
    assert fro < REL_FRO and row < REL_ROW, (fro, row)
    # Eq. 8: a dropped row leaves with the state it had entering its drop layer, bit for bit
    m1, m2 = masks[0][1], masks[1][1]
    entering1, _ = stack.forward(d["hidden"], d["positions"], d["cu_seqlens"], max(LENGTHS), upto=1)
    gone1 = torch.from_numpy(np.flatnonzero(~m1)).cuda()
    assert torch.equal(out[gone1], entering1[gone1])
    entering2, info2 = stack.forward(d["hidden"], d["positions"], d["cu_seqlens"], max(LENGTHS), drops=drops[:1],
                                     upto=2, G=G, n=n, A=A)
    assert np.array_equal(info2[0]["step"].token_keep.cpu().numpy().astype(bool), m1)
    gone2 = torch.from_numpy(np.flatnonzero(m1)[~m2]).cuda()
    assert gone2.numel() > 0
    assert torch.equal(out[gone2], entering2[gone2])
