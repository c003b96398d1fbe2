"""Parity of every CUDA entry point with the fp64 oracle on seeded inputs (GPU).

Small shapes that still span several 128-key tiles, ragged tails, empty requests, short requests
(N < n, N <= A + n), every supported d_k / G / n / head ratio, and the config-1 workload end to end.
"""
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


def _i32(x):
    return torch.tensor(np.asarray(x), dtype=torch.int32, device="cuda")


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------------------------------------ generator

def test_device_generator_matches_numpy_bitwise():
    w = recipe.small(lengths=(1000, 37, 3000), Hq=4, Hkv=2, dk=128, hdim=264, hot=("frac", 0.2), salt=41)
    host = gen.materialize(w)
    dev = sgpu.build_device(w, u=host["u"], hot_tok=host["hot_tok"])
    for k in ("Q", "K", "hidden"):
        got = dev[k].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, host[k]), k
    assert np.array_equal(dev["positions"].cpu().numpy(), host["positions"])
    assert np.array_equal(dev["slots"].cpu().numpy(), host["slots"])


# ------------------------------------------------------------------------------------------ selection

def _score_vectors(rng, lengths, G, kind):
    out = []
    for N in lengths:
        nb = -(-N // G)
        if kind == "zipf":
            v = 1.0 / np.arange(1, nb + 1) ** 1.2
            rng.shuffle(v)
        elif kind == "ties":
            v = rng.choice([0.0, 1.0, 2.0, 4.0], nb) / 8.0
        elif kind == "uniform":
            v = rng.random(nb)
        else:   # one dominant block
            v = rng.random(nb) * 1e-4
            if nb:
                v[rng.integers(nb)] = 1.0
        out.append(v.astype(np.float32))
    return out


@pytest.mark.parametrize("kind", ["zipf", "ties", "uniform", "dominant"])
@pytest.mark.parametrize("p", [0.5, 0.9, 0.99, 1.0])
def test_select_matches_oracle_on_the_same_scores(kind, p):
    rng = np.random.default_rng(hash((kind, p)) % 2**32)
    G, n, A = 64, 128, 128
    lengths = [5000, 0, 63, 200, 257, 64 * 8192, 1000]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    vecs = _score_vectors(rng, lengths, G, kind)
    scores = np.concatenate(vecs).astype(np.float32)
    cb = oracle.cu_blocks_of(cu, G)
    nb_cap = up.up_max_blocks(len(lengths), T, G)
    bs = torch.zeros(nb_cap, dtype=torch.float32, device="cuda")
    bs[:len(scores)] = torch.from_numpy(scores).cuda()
    bk = torch.zeros(nb_cap, dtype=torch.uint8, device="cuda")
    tk = torch.zeros(T, dtype=torch.uint8, device="cuda")
    ks = torch.zeros(len(lengths), dtype=torch.int32, device="cuda")
    st = _status()
    up.up_select_topp(bs, _i32(cb), _i32(cu), T, G, n, A, p, bk, tk, ks, st)
    assert up.up_read_status(st) == 0
    ref = oracle.select(scores.astype(np.float64), cu, G, n, A, p)
    assert np.array_equal(ks.cpu().numpy(), ref["kstar"])
    assert np.array_equal(bk.cpu().numpy()[:cb[-1]], ref["block_keep"])
    assert np.array_equal(tk.cpu().numpy(), ref["token_keep"])


def test_select_without_a_workspace_rejects_a_request_over_the_shared_memory_limit():
    G, N = 16, 16 * (up.MAX_BLOCKS_PER_REQUEST + 1)
    cu = np.array([0, N], dtype=np.int32)
    nb = up.up_max_blocks(1, N, G)
    bs = torch.ones(nb, device="cuda")
    st = _status()
    up.up_select_topp(bs, _i32(oracle.cu_blocks_of(cu, G)), _i32(cu), N, G, 128, 128, 0.9,
                      torch.zeros(nb, dtype=torch.uint8, device="cuda"), torch.zeros(N, dtype=torch.uint8, device="cuda"),
                      torch.zeros(1, dtype=torch.int32, device="cuda"), st)
    assert up.up_read_status(st) == 3


# requests of more than MAX_BLOCKS_PER_REQUEST blocks sort their keys through the workspace (tiles of
# 8192 keys); next to them, short requests take the shared-memory path in the same launch
@pytest.mark.parametrize("kind", ["zipf", "ties", "uniform", "dominant"])
@pytest.mark.parametrize("p", [0.5, 0.99, 1.0])
@pytest.mark.parametrize("G", [64, 16])
def test_select_beyond_the_shared_memory_limit_matches_oracle(kind, p, G):
    rng = np.random.default_rng(hash((kind, p, G, "large")) % 2**32)
    n, A = 128, 128
    if G == 64:
        lengths = [64 * 16384, 5000, 64 * 65536 + 17, 300, 64 * 8193]
    else:
        lengths = [16 * 20000 + 3, 0, 16 * 8192]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    scores = np.concatenate(_score_vectors(rng, lengths, G, kind)).astype(np.float32)
    cb = oracle.cu_blocks_of(cu, G)
    nb_cap = up.up_max_blocks(len(lengths), T, G)
    bs = torch.zeros(nb_cap, dtype=torch.float32, device="cuda")
    bs[:len(scores)] = torch.from_numpy(scores).cuda()
    ws = torch.empty(up.up_select_workspace_bytes(nb_cap), dtype=torch.uint8, device="cuda")
    ref = oracle.select(scores.astype(np.float64), cu, G, n, A, p)
    outs = []
    for _ in range(2):                       # deterministic, and nothing depends on the workspace's contents
        bk = torch.zeros(nb_cap, dtype=torch.uint8, device="cuda")
        tk = torch.zeros(T, dtype=torch.uint8, device="cuda")
        ks = torch.zeros(len(lengths), dtype=torch.int32, device="cuda")
        st = _status()
        up.up_select_topp(bs, _i32(cb), _i32(cu), T, G, n, A, p, bk, tk, ks, st, ws=ws)
        assert up.up_read_status(st) == 0
        assert np.array_equal(ks.cpu().numpy(), ref["kstar"])
        assert np.array_equal(bk.cpu().numpy()[:cb[-1]], ref["block_keep"])
        assert np.array_equal(tk.cpu().numpy(), ref["token_keep"])
        outs.append(tk)
        ws.fill_(0xAB)


# ------------------------------------------------------------------------------------------ compaction, Eq. 8, 16, 17

@pytest.mark.parametrize("keep_frac", [0.0, 0.3, 0.99, 1.0])
def test_compact_and_scatter_are_bit_exact(keep_frac):
    rng = np.random.default_rng(int(keep_frac * 100))
    lengths = [4500, 0, 17, 9000, 4096, 1]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, R, hdim = int(cu[-1]), len(lengths), 136
    keep = (rng.random(T) < keep_frac).astype(np.uint8)
    hidden = rng.integers(0, 2**16, (T, hdim)).astype(np.uint16)
    pos = rng.integers(0, 1 << 40, T)
    slots = rng.integers(0, 1 << 40, T)
    d_keep = torch.from_numpy(keep).cuda()
    d_hidden = torch.from_numpy(hidden.view(np.int16)).cuda().view(torch.bfloat16)
    d_pos, d_slots = torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda()
    L, layer = 3, 1
    outs = dict(kept_index=torch.zeros(T, dtype=torch.int32, device="cuda"),
                new_cu=torch.zeros(R + 1, dtype=torch.int32, device="cuda"),
                new_len=torch.zeros(R, dtype=torch.int32, device="cuda"),
                num_actual=torch.zeros(1, dtype=torch.int32, device="cuda"),
                out_hidden=torch.zeros(T, hdim, dtype=torch.bfloat16, device="cuda"),
                out_positions=torch.zeros(T, dtype=torch.int64, device="cuda"),
                out_slots=torch.zeros(T, dtype=torch.int64, device="cuda"),
                kept_len=torch.zeros(L, R, dtype=torch.int32, device="cuda"),
                drop_layer=torch.zeros(L, dtype=torch.uint8, device="cuda"))
    ws = torch.empty(up.up_compact_workspace_bytes(R, T), dtype=torch.uint8, device="cuda")
    st = _status()
    up.up_compact(d_keep, _i32(cu), outs["kept_index"], outs["new_cu"], outs["new_len"], outs["num_actual"], ws, st,
                  hidden=d_hidden, out_hidden=outs["out_hidden"], positions=d_pos, out_positions=outs["out_positions"],
                  slots=d_slots, out_slots=outs["out_slots"], kept_len=outs["kept_len"], drop_layer=outs["drop_layer"],
                  layer=layer)
    assert up.up_read_status(st) == 0
    got = {k: v.cpu().numpy() for k, v in outs.items() if k != "out_hidden"}
    got["num_actual"] = int(got["num_actual"][0])
    got["out_hidden"] = outs["out_hidden"].cpu().view(torch.int16).numpy().view(np.uint16)
    Tp = parity.check_compaction(got, keep, cu, hidden, pos, slots, layer=layer)
    # Eq. 8: new states = compacted rows + 1 (as raw bits) scattered into a copy of the block input
    new_states = (got["out_hidden"][:max(Tp, 1)].astype(np.uint32) + 1).astype(np.uint16)[:Tp]
    resid = d_hidden.clone()
    ns = torch.from_numpy(np.ascontiguousarray(new_states).view(np.int16)).cuda().view(torch.bfloat16)
    if Tp > 0:
        up.up_scatter_back(ns, outs["kept_index"], outs["num_actual"], resid, st)
    assert up.up_read_status(st) == 0
    expect = oracle.carry_forward(hidden, new_states, got["kept_index"][:Tp])
    assert np.array_equal(resid.cpu().view(torch.int16).numpy().view(np.uint16), expect)


def test_slot_mapping_eq16_matches_oracle():
    rng = np.random.default_rng(16)
    lengths = [300, 0, 1000, 17]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, R, B, mb = int(cu[-1]), len(lengths), 16, 70
    table = rng.permutation(R * mb).reshape(R, mb).astype(np.int32)
    pos = np.concatenate([np.sort(rng.choice(mb * B, L, replace=False)) for L in lengths]).astype(np.int64)
    slots = torch.zeros(T, dtype=torch.int64, device="cuda")
    st = _status()
    up.up_slot_mapping(torch.from_numpy(pos).cuda(), _i32(cu), _i32(table), B, slots, st)
    assert up.up_read_status(st) == 0
    assert np.array_equal(slots.cpu().numpy(), oracle.slot_mapping(pos, cu, table, B))
    # an out-of-table position is reported and written as -1
    pos[5] = mb * B
    up.up_slot_mapping(torch.from_numpy(pos).cuda(), _i32(cu), _i32(table), B, slots, st)
    assert up.up_read_status(st) == 5
    assert slots[5].item() == -1


def test_seqused_eq17_matches_oracle():
    rng = np.random.default_rng(17)
    L, R = 12, 9
    drop = (rng.random(L) < 0.4).astype(np.uint8)
    orig = rng.integers(100, 5000, R).astype(np.int32)
    kept = np.stack([(orig * rng.random(R)).astype(np.int32) for _ in range(L)])
    kv = (orig + rng.integers(0, 50, R)).astype(np.int32)
    out = torch.zeros(R, dtype=torch.int32, device="cuda")
    for layer in range(L):
        up.up_seqused(_i32(kept), torch.from_numpy(drop).cuda(), layer, _i32(orig), _i32(kv), out)
        assert np.array_equal(out.cpu().numpy(), oracle.seqused(kept, drop, layer, orig, kv)), layer


# ------------------------------------------------------------------------------------------ scoring

SCORE_CASES = [
    # Hq, Hkv, dk, G, n, lengths
    (8, 2, 128, 64, 128, (700, 1500, 90, 333)),
    (32, 8, 128, 64, 128, (2100,)),
    (4, 4, 64, 16, 32, (257, 1000, 0)),
    (16, 2, 256, 32, 128, (1100, 40)),
    (4, 2, 256, 128, 256, (900, 300)),
    (2, 1, 128, 64, 16, (50, 5, 0, 130)),
    (16, 8, 256, 64, 128, (2000, 513)),
    (8, 1, 64, 32, 1024, (3000, 1200)),
    # the score passes' work order on 152 SMs: 16 units per request (2 slabs x 8 KV heads) do not
    # divide the SMs, so the 2 slabs of a head form the CTA sets; 16 one-slab units, the plain order
    (32, 8, 128, 64, 256, (1300, 600)),
    (16, 16, 128, 64, 128, (900, 70, 1500)),
    # d_k = 256 with one job per key tile (the two epilogue pairs take alternate tiles), G = 16 (four
    # blocks per half-tile) and n = 64
    (8, 8, 256, 16, 128, (1500, 300)),
    (4, 2, 256, 64, 64, (700, 90, 1)),
]


def _run_score(w, host, with_tokens=True):
    d = sgpu.to_device(host)
    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n, A=w.A, p=w.p,
                       with_token_scores=with_tokens)
    step.score(d["Q"], d["K"])
    torch.cuda.synchronize()
    step.check()
    return step, d


# with per-token scores the call runs the two tcgen05 passes (row statistics, then recompute); without
# them, one pass that also writes per-row block sums, reduced after the row merge (slabs of 1, 2 or 4
# jobs of 128 rows; the other shapes keep two passes)
@pytest.mark.parametrize("tokens", [True, False], ids=["two_pass", "one_pass"])
@pytest.mark.parametrize("case", SCORE_CASES, ids=lambda c: "Hq%d_Hkv%d_dk%d_G%d_n%d" % c[:5])
def test_score_matches_oracle(case, tokens):
    Hq, Hkv, dk, G, n, lengths = case
    w = recipe.small(lengths=lengths, Hq=Hq, Hkv=Hkv, dk=dk, hdim=64, G=G, n=n, salt=50 + dk + G + n)
    host = gen.materialize(w, with_hidden=False)
    step, _ = _run_score(w, host, with_tokens=tokens)
    Q = gen.bf16_bits_to_f32(host["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(host["K"]).astype(np.float64)
    s_ref = oracle.token_scores(Q, K, host["cu_seqlens"], n)
    b_ref = oracle.block_scores_from_tokens(s_ref, host["cu_seqlens"], G)
    nbt = len(b_ref)
    parity.check_block_scores(step.block_scores.cpu().numpy()[:nbt], b_ref)
    if tokens:
        parity.check_block_scores(step.token_scores.cpu().numpy(), s_ref)


# up to 4,096 requests the one pass plans inside its single (fused) launch; beyond, a separate plan
# kernel searches the request offsets in global memory
@pytest.mark.parametrize("R", [4096, 4500])
def test_score_with_many_requests_matches_oracle(R):
    rng = np.random.default_rng(R)
    lengths = tuple(int(x) for x in rng.integers(0, 48, R))
    w = recipe.small(lengths=lengths, Hq=4, Hkv=2, dk=64, hdim=64, G=16, n=16, salt=R)
    host = gen.materialize(w, with_hidden=False)
    step, _ = _run_score(w, host, with_tokens=False)
    Q = gen.bf16_bits_to_f32(host["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(host["K"]).astype(np.float64)
    s_ref = oracle.token_scores(Q, K, host["cu_seqlens"], w.n)
    b_ref = oracle.block_scores_from_tokens(s_ref, host["cu_seqlens"], w.G)
    parity.check_block_scores(step.block_scores.cpu().numpy()[:len(b_ref)], b_ref)


@pytest.mark.parametrize("tokens", [True, False], ids=["two_pass", "one_pass"])
def test_score_closed_form_at_q_zero(tokens):
    """Q = 0: the scores follow the closed form 1/(n_eff) sum 1/(j+1) whatever K is (block scores: the
    closed form summed over the block and divided by G)."""
    G = 64
    w = recipe.small(lengths=(600, 77), Hq=4, Hkv=2, dk=128, hdim=64, G=G, n=128, salt=5)
    host = gen.materialize(w, with_hidden=False)
    host["Q"][:] = 0
    step, _ = _run_score(w, host, with_tokens=tokens)
    s = step.token_scores.cpu().numpy() if tokens else None
    b = step.block_scores.cpu().numpy()
    cu = host["cu_seqlens"]
    cb = oracle.cu_blocks_of(cu, G)
    for r in range(2):
        N = cu[r + 1] - cu[r]
        ne = min(128, N)
        exact = [sum(1.0 / (j + 1) for j in range(max(i, N - ne), N)) / ne for i in range(N)]
        if tokens:
            for i in range(N):
                assert abs(s[cu[r] + i] - exact[i]) <= 1e-4 * exact[i]
        for g in range(cb[r + 1] - cb[r]):
            eb = sum(exact[g * G:(g + 1) * G]) / G
            assert abs(b[cb[r] + g] - eb) <= 1e-4 * eb


@pytest.mark.parametrize("tokens", [True, False], ids=["two_pass", "one_pass"])
def test_score_is_deterministic_and_packing_invariant(tokens):
    w = recipe.small(lengths=(1500, 700, 2100), Hq=8, Hkv=2, dk=128, hdim=64, salt=61)
    host = gen.materialize(w, with_hidden=False)
    a, _ = _run_score(w, host, with_tokens=tokens)
    b, _ = _run_score(w, host, with_tokens=tokens)
    ba, bb = a.block_scores.cpu().numpy(), b.block_scores.cpu().numpy()
    assert np.array_equal(ba, bb)
    cu = host["cu_seqlens"]
    cb = oracle.cu_blocks_of(cu, w.G)
    for r in range(w.R):
        wr = w.replace(lengths=(w.lengths[r],))
        hr = dict(host)
        hr["cu_seqlens"] = np.array([0, w.lengths[r]], dtype=np.int32)
        hr["Q"] = host["Q"][cu[r]:cu[r + 1]]
        hr["K"] = host["K"][cu[r]:cu[r + 1]]
        sr, _ = _run_score(wr, hr, with_tokens=tokens)
        assert np.array_equal(sr.block_scores.cpu().numpy()[:cb[r + 1] - cb[r]], ba[cb[r]:cb[r + 1]]), r


def test_bad_cu_seqlens_is_reported_not_faulted():
    w = recipe.small(lengths=(500, 500), Hq=4, Hkv=2, dk=128, hdim=64, salt=3)
    host = gen.materialize(w, with_hidden=False)
    d = sgpu.to_device(host)
    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, 0, G=w.G, n=w.n)
    step.cu.copy_(_i32([0, 700, 600]))     # non-monotone
    step.score(d["Q"], d["K"])
    assert up.up_read_status(step.status) == 1


def test_bad_cu_seqlens_in_compaction_is_reported_and_stays_in_bounds():
    """Non-monotone cu_seqlens: up_compact reports UP_DEV_BAD_CU_SEQLENS and sets num_actual_tokens = 0;
    the token-side outputs, which do not depend on cu_seqlens, are the stable compaction of the mask."""
    w = recipe.small(lengths=(1500, 700, 900), Hq=4, Hkv=2, dk=128, hdim=64, salt=5)
    host = gen.materialize(w)
    d = sgpu.to_device(host)
    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n)
    keep = (np.random.default_rng(5).random(w.T) < 0.6).astype(np.uint8)
    step.token_keep.copy_(torch.from_numpy(keep).cuda())
    step.cu.copy_(_i32([0, 1600, 1500, w.T]))     # non-monotone
    step.compact(d["hidden"], d["positions"], d["slots"])
    torch.cuda.synchronize()
    assert up.up_read_status(step.status) == 1
    assert int(step.num_actual.item()) == 0
    ref = oracle.compact(keep, np.array([0, w.T], dtype=np.int32), host["hidden"], host["positions"],
                         host["slots"])
    Tp = ref["num_actual_tokens"]
    got = parity.step_to_numpy(step)
    assert np.array_equal(got["kept_index"][:Tp], ref["kept_index"])
    assert np.array_equal(got["out_hidden"][:Tp], ref["hidden"])
    assert np.array_equal(got["out_positions"][:Tp], ref["positions"])
    assert np.array_equal(got["out_slots"][:Tp], ref["slots"])


# ------------------------------------------------------------------------------------------ whole step

def test_config1_end_to_end():
    w = recipe.workload(1)
    host = gen.materialize(w)
    d = sgpu.to_device(host)
    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n, A=w.A, p=w.p, L=4, layer=2)
    resid = d["hidden"].clone()
    step.run(d["Q"], d["K"], d["hidden"], d["positions"], d["slots"], residual=resid)
    torch.cuda.synchronize()
    step.check()
    got = parity.step_to_numpy(step)
    Q = gen.bf16_bits_to_f32(host["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(host["K"]).astype(np.float64)
    ref = oracle.block_scores(Q, K, host["cu_seqlens"], w.G, w.n)
    parity.check_block_scores(got["block_scores"][:len(ref)], ref)
    nbound = parity.check_selection(got["block_keep"][:len(ref)], got["token_keep"], ref, host["cu_seqlens"],
                                    w.G, w.n, w.A, w.p)
    parity.check_compaction(got, got["token_keep"], host["cu_seqlens"], host["hidden"], host["positions"],
                            host["slots"], layer=2)
    assert np.array_equal(resid.cpu().view(torch.int16).numpy().view(np.uint16), host["hidden"])
    print(f"config 1: k*={got['kstar'].tolist()} kept={got['num_actual']}/{w.T} boundary={nbound}")
