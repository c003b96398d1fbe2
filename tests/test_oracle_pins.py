"""Pins of the fp64 oracle against facts fixed by the paper and by mathematics.

Paper: "UniPrefill: Universal Long-Context Prefill Acceleration via Block-wise
Dynamic Sparsification" (arXiv 2605.06221).  None of these tests re-derives an
expected value by calling the oracle's own formula: each expected value is a
closed form, a library routine on a special case, a brute-force enumeration,
an invariant, or a hand-worked fixture under tests/golden/.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from synth import cpu as gen
from synth import recipe


def _small_inputs(lengths=(300, 129, 64, 7, 1000), Hq=4, Hkv=2, dk=64, seed=3, salt=5, n=128, G=64):
    w = recipe.small(lengths=lengths, Hq=Hq, Hkv=Hkv, dk=dk, n=n, G=G, seed=seed, salt=salt)
    d = gen.materialize(w, with_hidden=False)
    Q = gen.bf16_bits_to_f32(d["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(d["K"]).astype(np.float64)
    return w, Q, K, d["cu_seqlens"]


# ------------------------------------------------------------------------------- scoring (Eqs. 2-4)

@pytest.mark.parametrize("G", [16, 64, 128])
def test_block_mass_sums_to_one_over_G(G):
    """Every causal softmax row sums to 1, so with the head mean sum_g b_g = 1/G exactly (Eq. 4, R2, R4)."""
    w, Q, K, cu = _small_inputs(G=G)
    bs = oracle.block_scores(Q, K, cu, G, w.n)
    cb = oracle.cu_blocks_of(cu, G)
    for r in range(len(cu) - 1):
        tot = bs[cb[r]:cb[r + 1]].sum()
        assert abs(tot - 1.0 / G) < 1e-12


@pytest.mark.parametrize("N,n", [(50, 16), (10, 16), (130, 128), (64, 64)])
def test_closed_form_at_q_zero(N, n):
    """Q = 0 makes every visible logit 0: the row at local position j spreads 1/(j+1) over keys 0..j,
    so s_i = (1/n_eff) * sum_{j=max(i, N-n_eff)}^{N-1} 1/(j+1) exactly (Eqs. 2-3 with the causal window)."""
    rng = np.random.default_rng(0)
    Hq, Hkv, dk = 4, 2, 32
    Q = np.zeros((N, Hq, dk))
    K = rng.standard_normal((N, Hkv, dk))
    s = oracle.token_scores(Q, K, [0, N], n)
    ne = min(n, N)
    for i in range(N):
        exact = sum(Fraction(1, j + 1) for j in range(max(i, N - ne), N)) / ne
        assert abs(s[i] - float(exact)) < 1e-13, i


def test_gqa_equals_explicit_head_expansion():
    """Grouped-query sharing (R3) equals repeating each KV head `group` times consecutively."""
    w, Q, K, cu = _small_inputs(Hq=8, Hkv=2)
    s = oracle.token_scores(Q, K, cu, w.n)
    s_rep = oracle.token_scores(Q, np.repeat(K, 4, axis=1), cu, w.n)
    np.testing.assert_allclose(s, s_rep, rtol=0, atol=1e-15)


@pytest.mark.parametrize("N", [1, 5, 33])
def test_reduces_to_library_causal_attention_when_window_is_whole_sequence(N):
    """With n = N the window is the whole request; the attention matrix is then what
    torch's scaled_dot_product_attention (causal, default 1/sqrt(d) scale) returns for V = I."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(N)
    Hq, Hkv, dk = 3, 1, 16
    Q = rng.standard_normal((N, Hq, dk))
    K = rng.standard_normal((N, Hkv, dk))
    s = oracle.token_scores(Q, K, [0, N], N)
    expect = np.zeros(N)
    for h in range(Hq):
        q = torch.tensor(Q[:, h, :])[None, None]
        k = torch.tensor(K[:, 0, :])[None, None]
        eye = torch.eye(N, dtype=torch.float64)[None, None]
        A = torch.nn.functional.scaled_dot_product_attention(q, k, eye, is_causal=True)[0, 0].numpy()
        expect += A.sum(axis=0)
    expect /= N * Hq
    np.testing.assert_allclose(s, expect, rtol=1e-12, atol=1e-15)


def test_single_dominant_key_takes_the_mass_of_later_rows():
    """All window queries equal q; key i0 = 40 q/|q| dominates every row j >= i0 (Eq. 2)."""
    rng = np.random.default_rng(7)
    N, n, dk = 200, 32, 64
    q = rng.standard_normal(dk)
    Q = np.tile(q, (N, 1, 1)).reshape(N, 1, dk)
    K = rng.standard_normal((N, 1, dk)) * 0.1
    i0 = 180
    K[i0, 0] = 40.0 * q / np.linalg.norm(q)
    s = oracle.token_scores(Q, K, [0, N], n)
    rows_after = N - i0                       # window rows j with j >= i0
    assert s[i0] > 0.999 * rows_after / n
    assert s[i0] <= rows_after / n + 1e-12


# ------------------------------------------------------------------------------- selection (Eq. 5, Eq. 14)

def _golden(name):
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("topp_cases.json")["cases"], ids=lambda c: c["name"])
def test_topp_golden(case):
    b = np.asarray(case["scores_x64"], dtype=np.float64) / 64.0
    d = oracle.select_request(b, case["N"], case["G"], case["n"], case["A"], case["p"])
    assert d["kstar"] == case["kstar"]
    assert sorted(np.flatnonzero(d["ranked"]).tolist()) == case["ranked"]
    assert d["token_keep"].astype(int).tolist() == case["token_keep"]
    assert d["block_keep"].astype(int).tolist() == case["block_keep"]


def test_phi_golden():
    g = _golden("eq14_phi.json")
    for e in g["phi"]:
        x = np.float32(float(e["x"]))
        assert int(x.view(np.uint32)) == int(e["bits"], 16)
        assert int(oracle.phi(np.array([x]))[0]) == int(e["phi"], 16), e
    for e in g["packed"]:
        got = int(oracle.pack_key(np.array([np.float32(float(e["x"]))]), np.array([e["g"]]))[0])
        assert got == int(e["packed"], 16)


def test_phi_is_monotone_on_every_float_class_but_negative_zero():
    """Eq. 14: sorting phi(x) as unsigned integers orders floats like a comparison sort."""
    rng = np.random.default_rng(11)
    special = np.array([0.0, 1e-45, 3e-45, 1.1754942e-38, 1.17549435e-38, 1.0, 3.4028235e38, np.inf,
                        -1e-45, -1.1754942e-38, -1.0, -3.4028235e38, -np.inf, 0.5, -0.5], dtype=np.float32)
    rand = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-40, 38, 4000).astype(np.float32),
        (rng.integers(0, 2**23, 1000).astype(np.uint32)).view(np.float32),            # positive denormals
        (rng.integers(0, 2**23, 1000).astype(np.uint32) | np.uint32(0x80000000)).view(np.float32)])
    x = np.unique(np.concatenate([special, rand[np.isfinite(rand) | np.isinf(rand)]]))
    x = x[~((x == 0) & np.signbit(x))]
    ph = oracle.phi(x).astype(np.uint64)
    assert np.all(np.diff(ph.astype(np.int64)) > 0)       # x is sorted ascending, so phi must be too
    # the literal comparison maps -0.0 below every negative number (the reachable scores are >= +0)
    assert int(oracle.phi(np.array([-0.0], dtype=np.float32))[0]) == 0
    assert int(oracle.phi(np.array([-1e-45], dtype=np.float32))[0]) > 0


def test_packed_key_order_matches_rank_order():
    """Sorting Eq. 14's packed words descending gives Eq. 5's permutation with R6's tie rule."""
    rng = np.random.default_rng(5)
    for _ in range(50):
        nb = int(rng.integers(1, 300))
        b = rng.choice(np.array([0.0, 1e-30, 0.25, 0.5, 1e-7, 3.0], dtype=np.float32), nb)
        b = np.where(rng.random(nb) < 0.5, b, rng.random(nb).astype(np.float32))
        keys = oracle.pack_key(b, np.arange(nb))
        by_key = np.argsort(keys)[::-1]
        assert np.array_equal(by_key, oracle.rank_order(b.astype(np.float64)))


def _min_subset_size(b, thr):
    nb = len(b)
    for k in range(0, nb + 1):
        for comb in itertools.combinations(range(nb), k):
            if sum(b[list(comb)]) >= thr:
                return k
    return None


@pytest.mark.parametrize("seed", range(40))
def test_kstar_is_the_minimal_subset_size_by_enumeration(seed):
    """Eq. 5's k* is the size of the smallest block subset of mass >= p * total (brute force, nb <= 10)."""
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(1, 11))
    b = rng.integers(0, 9, nb).astype(np.float64) / 8.0 if seed % 3 == 0 else rng.random(nb) ** 3
    if b.sum() == 0:
        b[0] = 1.0
    p = float(rng.choice([0.5, 0.8, 0.9, 0.99, 1.0]))
    order, kstar = oracle.topp_kstar(b, p)
    total = math.fsum(b)
    thr = p * total
    assert kstar == _min_subset_size(b, thr - 1e-12 * total)
    kept = math.fsum(b[order[:kstar]])
    assert kept >= thr - 1e-12 * total
    if kstar > 1:
        assert math.fsum(b[order[:kstar - 1]]) < thr + 1e-12 * total   # minimality


@pytest.mark.parametrize("p", [0.9, 0.98, 0.99])
def test_dropped_mass_bound_eq6(p):
    """Eq. 6: the dropped blocks hold at most (1 - p) of the mass; sinks and window are kept."""
    w, Q, K, cu = _small_inputs(lengths=(2000, 700, 130), n=128, G=64)
    bs = oracle.block_scores(Q, K, cu, 64, 128)
    sel = oracle.select(bs, cu, 64, 128, 128, p)
    cb = sel["cu_blocks"]
    for r in range(len(cu) - 1):
        b = bs[cb[r]:cb[r + 1]]
        ranked = sel["ranked"][cb[r]:cb[r + 1]].astype(bool)
        assert b[~ranked].sum() <= (1 - p) * b.sum() + 1e-15
        N = cu[r + 1] - cu[r]
        tk = sel["token_keep"][cu[r]:cu[r + 1]]
        assert tk[:min(128, N)].all() and tk[max(0, N - 128):].all()


# ------------------------------------------------------------------------------- compaction, Eq. 8, Eq. 16, Eq. 17

def test_compaction_invariants():
    rng = np.random.default_rng(2)
    cu = np.array([0, 100, 100, 357, 400])
    keep = (rng.random(400) < 0.6).astype(np.uint8)
    hidden = rng.integers(0, 2**16, (400, 24)).astype(np.uint16)
    pos = rng.integers(0, 1 << 40, 400)
    c = oracle.compact(keep, cu, hidden, pos, pos + 1)
    ki = c["kept_index"]
    assert len(ki) == keep.sum() == c["num_actual_tokens"]
    assert np.all(np.diff(ki) > 0)                      # stable (ascending) order
    assert keep[ki].all()
    others = np.setdiff1d(np.arange(400), ki)
    assert not keep[others].any()                       # every kept token is present
    assert np.array_equal(c["hidden"], hidden[ki])
    nc = c["new_cu_seqlens"]
    assert nc[0] == 0 and nc[-1] == keep.sum() and np.all(np.diff(nc) >= 0)
    for r in range(4):                                   # request r's kept tokens sit in [nc[r], nc[r+1])
        seg = ki[nc[r]:nc[r + 1]]
        assert np.all((seg >= cu[r]) & (seg < cu[r + 1]))


def test_eq8_identities():
    rng = np.random.default_rng(4)
    H = rng.integers(0, 2**16, (300, 16)).astype(np.uint16)
    keep = (rng.random(300) < 0.7).astype(np.uint8)
    c = oracle.compact(keep, [0, 300], H)
    assert np.array_equal(oracle.carry_forward(H, c["hidden"], c["kept_index"]), H)   # identity sublayers
    newk = (c["hidden"] + 1).astype(np.uint16)
    out = oracle.carry_forward(H, newk, c["kept_index"])
    assert np.array_equal(out[keep == 0], H[keep == 0])                                # dropped rows carried
    assert np.array_equal(out[keep == 1], newk)                                        # kept rows updated


def test_eq16_golden():
    g = _golden("eq16_eq17.json")["eq16"]
    got = oracle.slot_mapping(g["positions"], g["cu_seqlens"], g["block_table"], g["B"])
    assert got.tolist() == g["slots"]


def test_eq17_golden():
    g = _golden("eq16_eq17.json")["eq17"]
    for layer, expect in enumerate(g["seqused"]):
        got = oracle.seqused(g["kept_len"], g["drop_layer"], layer, g["orig_len"], g["kv_len"])
        assert got.tolist() == expect, layer


def test_full_step_on_planted_workload_keeps_hot_blocks():
    """On a small planted workload the hot blocks carry extra mass and all are ranked.

    The shift of 2.0 along the unit mean window query moves a logit by about
    2 * (q . u) / sqrt(d_k), i.e. ~0.1 on average: a weak but systematic signal."""
    w = recipe.small(lengths=(4096,), Hq=8, Hkv=2, dk=128, hot=("count", 6), salt=23)
    d = gen.materialize(w, with_hidden=False)
    Q = gen.bf16_bits_to_f32(d["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(d["K"]).astype(np.float64)
    out = oracle.drop_step(Q, K, d["cu_seqlens"], w.G, w.n, w.A, w.p)
    bs = out["block_scores"]
    hot = d["hot"][0]
    cold = [g for g in range(len(bs)) if g not in hot and g > 2 and g < len(bs) - 3]
    assert np.mean(bs[hot]) > 1.05 * np.median(bs[cold])
    assert all(out["ranked"][g] for g in hot)
