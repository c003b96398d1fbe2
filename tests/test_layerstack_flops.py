"""FLOPs accounting of the decoder stack that consumes the drop step (CPU): UniPrefill section 3.3,
"FLOPs analysis", Eqs. 9-10.

The accounting is pinned twice: against a brute-force count of every matmul the float64 recomputation
of the stack performs (torch's FLOP counter, causal attention row by row so that it does exactly the
visible work), and against the closed forms of Eq. 10 (one drop) and Eq. 9 (two drops), for the
linear (projection) part whose cost per layer is proportional to the tokens it sees.
"""
import numpy as np
import pytest
import torch
from torch.utils.flop_counter import FlopCounterMode

from long_context_prefill_varlen_gb300 import layerstack as ls
from tests import stack_ref

TINY = ls.StackGeometry(d=32, Hq=4, Hkv=2, dk=8, ffn=48)


def _stack(L):
    return ls.RandomLlamaStack(L, TINY, seed=3, device="cpu", init_device="cpu")


def _keep_mask(lengths, frac, seed):
    rng = np.random.default_rng(seed)
    return rng.random(int(sum(lengths))) < frac


def _kept_lengths(lengths, keep):
    cu = np.concatenate([[0], np.cumsum(lengths)])
    return [int(keep[cu[r]:cu[r + 1]].sum()) for r in range(len(lengths))]


@pytest.mark.parametrize("drop_layers", [(), (1,), (0, 2)])
def test_accounting_equals_a_brute_force_count_of_the_recomputation(drop_layers):
    lengths = [37, 0, 64, 21]
    L = 4
    stack = _stack(L)
    T = sum(lengths)
    h = torch.randn(T, TINY.d, generator=torch.Generator().manual_seed(1), dtype=torch.float64)
    pos = np.concatenate([np.arange(N) for N in lengths]).astype(np.int64)
    drops, cur = [], lengths
    for i, layer in enumerate(drop_layers):
        keep = _keep_mask(cur, 0.6, 10 + i)
        drops.append((layer, keep))
        cur = _kept_lengths(cur, keep)
    with FlopCounterMode(display=False) as fc:
        stack_ref.forward(stack, h, pos, lengths, drops, rowwise=True)
    counted = fc.get_total_flops()
    kept_per_drop = []
    cur = lengths
    for layer, keep in drops:
        cur = _kept_lengths(cur, keep)
        kept_per_drop.append((layer, cur))
    assert counted == ls.stack_flops(lengths, TINY, L, kept_per_drop)


def test_one_drop_saves_eq10_on_the_projections():
    """Eq. 10: a drop at layer l1 with retention rho saves (1 - rho) x (layers after l1) x the per-layer
    projection cost of the whole stream; with 0-based layers the FFN of l1 itself is also saved (it is a
    sublayer after the scoring attention)."""
    g = ls.LLAMA_3_1_8B
    lengths = [32768]
    L, l1 = 32, 10
    for rho in (1.0, 0.99, 0.5, 0.25):
        kept = [int(round(rho * 32768))]
        rho_exact = kept[0] / 32768
        full = ls.stack_flops(lengths, g, L)
        drop = ls.stack_flops(lengths, g, L, [(l1, kept)])
        attn_saved = (L - 1 - l1) * (ls.attention_flops(lengths, g) - ls.attention_flops(kept, g))
        per_tok_layer = ls.linear_flops_per_token(g)
        per_tok_ffn = ls.linear_flops_per_token(g, attention=False)
        eq10 = (1 - rho_exact) * 32768 * ((L - 1 - l1) * per_tok_layer + per_tok_ffn)
        assert full - drop - attn_saved == pytest.approx(eq10, rel=1e-12)
        if rho == 1.0:
            assert full == drop


def test_two_drops_save_eq9_with_each_rho_relative_to_the_stream_it_drops_from():
    """Eq. 9, read with rho_k the k-th drop's own retention and FLOPs_l(N) the cost of layer l on the
    stream that drop is applied to: the projection savings add up exactly."""
    g = ls.StackGeometry(d=512, Hq=8, Hkv=2, dk=64, ffn=1536)
    L, (l1, l2) = 12, (3, 7)
    N0 = [4000, 1000]
    N1 = [3000, 700]
    N2 = [1500, 650]
    full = ls.stack_flops(N0, g, L)
    drop = ls.stack_flops(N0, g, L, [(l1, N1), (l2, N2)])
    attn_saved = ((l2 - l1) * (ls.attention_flops(N0, g) - ls.attention_flops(N1, g))
                  + (L - 1 - l2) * (ls.attention_flops(N0, g) - ls.attention_flops(N2, g)))
    c, cf = ls.linear_flops_per_token(g), ls.linear_flops_per_token(g, attention=False)
    T0, T1, T2 = sum(N0), sum(N1), sum(N2)
    rho1, rho2 = T1 / T0, T2 / T1
    eq9 = (1 - rho1) * T0 * ((L - 1 - l1) * c + cf) + (1 - rho2) * T1 * ((L - 1 - l2) * c + cf)
    assert full - drop - attn_saved == pytest.approx(eq9, rel=1e-12)


def test_drop_layers_must_increase():
    with pytest.raises(ValueError):
        ls.stack_flops([100], TINY, 4, [(2, [50]), (1, [20])])


def test_recomputation_invariants():
    """The row-by-row and the masked-square attention agree; a drop that keeps every token is the
    identity (Eq. 8 with an empty dropped set); a dropped row leaves the stack with the state it had
    entering the drop layer."""
    lengths = [30, 45, 0, 12]
    L = 3
    stack = _stack(L)
    T = sum(lengths)
    h = torch.randn(T, TINY.d, generator=torch.Generator().manual_seed(2), dtype=torch.float64)
    pos = np.concatenate([np.arange(N) for N in lengths]).astype(np.int64)
    a = stack_ref.forward(stack, h, pos, lengths, rowwise=True)
    b = stack_ref.forward(stack, h, pos, lengths)
    assert torch.allclose(a, b, rtol=1e-12, atol=1e-12)
    c = stack_ref.forward(stack, h, pos, lengths, [(1, np.ones(T, dtype=bool))])
    assert torch.allclose(b, c, rtol=1e-12, atol=1e-12)
    keep = _keep_mask(lengths, 0.5, 4)
    d = stack_ref.forward(stack, h, pos, lengths, [(1, keep)])
    entering = stack_ref.forward(stack, h, pos, lengths, upto=1)
    assert torch.equal(d[torch.from_numpy(~keep)], entering[torch.from_numpy(~keep)])
    assert not torch.allclose(d[torch.from_numpy(keep)], b[torch.from_numpy(keep)])
