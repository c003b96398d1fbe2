"""The bounds-checked build of the library (GPU).

libuniprefill_debug.so is the library compiled with -DUP_DEBUG_BOUNDS: every kernel checks each global
index against the length of its array, records UP_DEV_BOUNDS in the status word on a violation and
skips the access.  It stands in for a memory checker: the parity cases of every entry point run through
it here, must leave every status word at 0, and must give outputs bit-identical to the normal build's.
"""
import contextlib

import numpy as np
import pytest
import torch

import long_context_prefill_varlen_gb300 as up
from long_context_prefill_varlen_gb300 import _build
from synth import cpu as gen
from synth import gpu as sgpu
from synth import recipe

pytestmark = pytest.mark.gpu

# Hq, Hkv, dk, G, n, lengths: jobs of 1, 2, 4 and 8 per tile (and 1 at d_k = 256), every G, and streams of at most 8, at
# most 64 and more than 64 tiles of 1,024 tokens for the compaction's three launch paths
CASES = [
    (8, 2, 128, 64, 128, (700, 1500, 90, 333)),
    (4, 4, 64, 16, 32, (257, 1000, 0)),
    (16, 2, 256, 32, 128, (1100, 40)),
    (8, 1, 64, 32, 1024, (3000, 1200)),
    (4, 2, 256, 128, 256, (900, 300)),
    (2, 1, 64, 64, 128, (9000, 1, 2500)),
    (2, 1, 64, 64, 128, (70000, 500)),
    (4, 4, 256, 16, 64, (1200, 70)),
]


@contextlib.contextmanager
def library(path):
    """The binding's calls go to the library at `path` inside the block."""
    saved = up._lib
    try:
        up._lib = None
        up.load_library(path)
        yield
    finally:
        up._lib = saved


@pytest.fixture(scope="module")
def debug_lib():
    return _build.build(debug_bounds=True)


def _run(w, host, tokens):
    d = sgpu.to_device(host)
    L = 3
    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n, A=w.A, p=w.p, L=L, layer=1,
                       with_token_scores=tokens)
    step.run(d["Q"], d["K"], d["hidden"], d["positions"], d["slots"])
    new_states = (step.out_hidden.view(torch.int16) ^ 1).view(torch.bfloat16)
    residual = d["hidden"].clone()
    step.scatter_back(new_states, residual)
    B, mb = 16, max(1, -(-max(w.lengths) // 16))
    rng = np.random.default_rng(7)
    table = torch.from_numpy(rng.permutation(w.R * mb).reshape(w.R, mb).astype(np.int32)).cuda()
    slots = torch.zeros(max(1, w.T), dtype=torch.int64, device="cuda")
    up.up_slot_mapping(step.out_positions[:w.T], step.new_cu, table, B, slots, step.status, num_tokens=step.num_actual)
    orig = torch.tensor(w.lengths, dtype=torch.int32, device="cuda")
    seq = step.seqused(orig, orig + 3, 2).clone()
    torch.cuda.synchronize()
    status = up.up_read_status(step.status)
    n = int(step.num_actual.item())
    out = dict(block_scores=step.block_scores, block_keep=step.block_keep, token_keep=step.token_keep,
               kstar=step.kstar, kept_index=step.kept_index[:n], new_cu=step.new_cu, kept_len=step.kept_len,
               out_hidden=step.out_hidden[:n].view(torch.int16), out_positions=step.out_positions[:n],
               out_slots=step.out_slots[:n], residual=residual.view(torch.int16), slots=slots[:n], seqused=seq)
    if tokens:
        out["token_scores"] = step.token_scores
    return status, {k: v.cpu() for k, v in out.items()}


@pytest.mark.parametrize("tokens", [False, True], ids=["one_pass", "two_pass"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "Hq%d_Hkv%d_dk%d_G%d_n%d_T%d" % (c[:5] + (sum(c[5]),)))
def test_bounds_checked_build_runs_the_step_clean_and_identical(case, tokens, debug_lib):
    Hq, Hkv, dk, G, n, lengths = case
    w = recipe.small(lengths=lengths, Hq=Hq, Hkv=Hkv, dk=dk, hdim=64, G=G, n=n, p=0.9, salt=90 + dk + G + n)
    host = gen.materialize(w)
    assert up.up_debug_bounds() == 0
    st_ref, ref = _run(w, host, tokens)
    with library(debug_lib):
        assert up.up_debug_bounds() == 1
        st_dbg, got = _run(w, host, tokens)
    assert st_ref == 0 and st_dbg == 0, (st_ref, st_dbg)
    for k in ref:
        assert torch.equal(ref[k], got[k]), k


def test_bounds_checked_build_selects_a_request_beyond_shared_memory(debug_lib):
    G, n, A, p = 16, 128, 128, 0.95
    lengths = [16 * 9000 + 5, 3000]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    nb_cap = up.up_max_blocks(len(lengths), T, G)
    rng = np.random.default_rng(3)
    bs = torch.from_numpy((1.0 / np.arange(1, nb_cap + 1) ** 1.1)[rng.permutation(nb_cap)].astype(np.float32)).cuda()
    cb = torch.tensor([0, -(-lengths[0] // G), -(-lengths[0] // G) + -(-lengths[1] // G)], dtype=torch.int32).cuda()
    cu_d = torch.from_numpy(cu).cuda()

    def run():
        ws = torch.empty(up.up_select_workspace_bytes(nb_cap), dtype=torch.uint8, device="cuda")
        bk = torch.zeros(nb_cap, dtype=torch.uint8, device="cuda")
        tk = torch.zeros(T, dtype=torch.uint8, device="cuda")
        ks = torch.zeros(len(lengths), dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        up.up_select_topp(bs, cb, cu_d, T, G, n, A, p, bk, tk, ks, st, ws=ws)
        return up.up_read_status(st), bk.cpu(), tk.cpu(), ks.cpu()

    ref = run()
    with library(debug_lib):
        got = run()
    assert ref[0] == 0 and got[0] == 0
    for a, b in zip(ref[1:], got[1:]):
        assert torch.equal(a, b)


def test_bounds_checked_build_compacts_without_a_workspace(debug_lib):
    rng = np.random.default_rng(11)
    lengths = [66000, 7, 1500]
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).cuda()
    T, R, hdim = sum(lengths), len(lengths), 64
    keep = torch.from_numpy((rng.random(T) < 0.4).astype(np.uint8)).cuda()
    hidden = torch.from_numpy(rng.integers(0, 2**16, (T, hdim)).astype(np.uint16).view(np.int16)).cuda()

    def run():
        i32 = dict(dtype=torch.int32, device="cuda")
        o = dict(ki=torch.zeros(T, **i32), cu=torch.zeros(R + 1, **i32), ln=torch.zeros(R, **i32),
                 na=torch.zeros(1, **i32), oh=torch.zeros(T, hdim, dtype=torch.bfloat16, device="cuda"),
                 st=torch.zeros(1, **i32))
        up.up_compact_noalloc(keep, cu, o["ki"], o["cu"], o["ln"], o["na"], o["st"], hidden=hidden.view(torch.bfloat16),
                              out_hidden=o["oh"])
        o["oh"] = o["oh"].view(torch.int16)            # bit patterns (random bits include NaNs)
        return up.up_read_status(o["st"]), {k: v.cpu() for k, v in o.items() if k != "st"}

    ref = run()
    with library(debug_lib):
        got = run()
    assert ref[0] == 0 and got[0] == 0
    for k in ref[1]:
        assert torch.equal(ref[1][k], got[1][k]), k
