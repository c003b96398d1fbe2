"""The allocation-free compaction entry point, up_compact_noalloc, against up_compact (GPU).

Some callers cannot give this library device scratch memory: an engine whose memory planner owns all
device memory once it has started, a plugin host that only hands over the tensors it already holds,
or a loop that must not pay cudaMalloc's implicit synchronisation.  up_compact_noalloc serves them with
a fixed scratch array built into the library.  This file checks, through the C ABI, that it returns
exactly what the workspace version returns (compaction is bit-exact) and what the fp64 oracle's
compaction gives, on calls in a row so that whatever one call leaves in the shared array cannot leak
into the next.  The streams take every launch path of the compaction through the shared array: at
most 8 tiles of 1,024 tokens (one launch that scans the stream itself), up to 64 tiles (the scan
kernel counts the tiles) and more than 64 tiles (a separate count kernel writes the tile counts).
It runs last.
"""
import ctypes

import numpy as np
import pytest
import torch

import long_context_prefill_varlen_gb300 as up
from tests import parity

pytestmark = pytest.mark.gpu


def _case(seed, keep_frac, lengths, hdim=264):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    return dict(
        cu=torch.from_numpy(cu).cuda(),
        keep=torch.from_numpy((rng.random(T) < keep_frac).astype(np.uint8)).cuda(),
        hidden=torch.from_numpy(rng.integers(0, 2**16, (T, hdim)).astype(np.uint16).view(np.int16)).cuda()
        .view(torch.bfloat16),
        pos=torch.from_numpy(rng.integers(0, 1 << 40, T)).cuda(),
        slots=torch.from_numpy(rng.integers(0, 1 << 40, T)).cuda(),
        T=T, R=len(lengths), hdim=hdim)


def _outputs(c, L=3):
    T, R = c["T"], c["R"]
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(kept_index=torch.full((T,), -7, **i32), new_cu=torch.full((R + 1,), -7, **i32),
                new_len=torch.full((R,), -7, **i32), num_actual=torch.full((1,), -7, **i32),
                out_hidden=torch.zeros(T, c["hdim"], dtype=torch.bfloat16, device="cuda"),
                out_pos=torch.zeros(T, dtype=torch.int64, device="cuda"),
                out_slots=torch.zeros(T, dtype=torch.int64, device="cuda"),
                kept_len=torch.zeros(L, R, **i32), drop_layer=torch.zeros(L, dtype=torch.uint8, device="cuda"),
                status=torch.zeros(1, **i32))


def _run(c, noalloc):
    o = _outputs(c)
    kw = dict(hidden=c["hidden"], out_hidden=o["out_hidden"], positions=c["pos"], out_positions=o["out_pos"],
              slots=c["slots"], out_slots=o["out_slots"], kept_len=o["kept_len"], drop_layer=o["drop_layer"], layer=1)
    if noalloc:
        up.up_compact_noalloc(c["keep"], c["cu"], o["kept_index"], o["new_cu"], o["new_len"], o["num_actual"],
                              o["status"], **kw)
    else:
        ws = torch.empty(up.up_compact_workspace_bytes(c["R"], c["T"]), dtype=torch.uint8, device="cuda")
        up.up_compact(c["keep"], c["cu"], o["kept_index"], o["new_cu"], o["new_len"], o["num_actual"], ws,
                      o["status"], **kw)
    assert up.up_read_status(o["status"]) == 0
    n = int(o["num_actual"].item())
    res = {k: v.cpu() for k, v in o.items()}
    for k in ("kept_index", "out_hidden", "out_pos", "out_slots"):
        res[k] = res[k][:n]
    res["out_hidden"] = res["out_hidden"].view(torch.int16)
    return res


def _against_oracle(c, got):
    """the noalloc outputs, bit-exact against the oracle's compaction of the same mask and inputs"""
    n = int(got["num_actual"][0])
    kl = got["kept_len"].numpy()
    g = dict(num_actual=n, kept_index=got["kept_index"].numpy(), new_cu=got["new_cu"].numpy(),
             new_len=got["new_len"].numpy(), out_hidden=got["out_hidden"].numpy().view(np.uint16),
             out_positions=got["out_pos"].numpy(), out_slots=got["out_slots"].numpy(), kept_len=kl,
             drop_layer=got["drop_layer"].numpy())
    parity.check_compaction(g, c["keep"].cpu().numpy(), c["cu"].cpu().numpy(),
                            hidden=c["hidden"].cpu().view(torch.int16).numpy().view(np.uint16),
                            positions=c["pos"].cpu().numpy(), slots=c["slots"].cpu().numpy(), layer=1)


def test_noalloc_matches_the_workspace_version_and_the_oracle_on_calls_in_a_row():
    cases = [_case(1, 0.7, [5000, 0, 37, 12000, 1025]),      # 18 tiles: the scan kernel counts the tiles
             _case(2, 0.25, [3000, 9000, 1, 4096]),          # 16 tiles
             _case(3, 0.5, [70000, 3, 1200], hdim=64),       # 70 tiles: separate count kernel
             _case(4, 0.9, [2000, 0, 4100, 1], hdim=64),     # 6 tiles: the one-launch path
             _case(5, 0.1, [66000, 50], hdim=64)]            # 65 tiles again, after a short stream
    for c in cases:
        ref = _run(c, noalloc=False)
        got = _run(c, noalloc=True)
        for k in ref:
            assert torch.equal(ref[k], got[k]), k
        _against_oracle(c, got)


def test_noalloc_rejects_more_tokens_than_its_scratch_holds():
    lib = up.load_library()
    fake = ctypes.c_void_p(0x1000)        # never dereferenced: the size check comes first
    T = up.NOALLOC_MAX_TOKENS + 1
    code = lib.up_compact_noalloc(fake, fake, 1, T, None, 0, None, None, None, None, None, fake, fake, fake, fake,
                                  None, None, 0, 0, fake, None)
    assert code == up.UP_ERR_WORKSPACE
