"""The C-ABI library loads on a host without a GPU, exports every declared entry point, and rejects
bad host-side arguments before touching the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "uniprefill.h")


@pytest.fixture(scope="module")
def lib():
    from long_context_prefill_varlen_gb300 import _build
    _build.build()
    import long_context_prefill_varlen_gb300 as up
    return up.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(up_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    # and nothing exported with the prefix is undeclared
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    exported = set(re.findall(r" T (up_[a-z_0-9]+)", out))
    assert exported == set(names)


def test_sizing_helpers(lib):
    import long_context_prefill_varlen_gb300 as up
    assert up.up_abi_version() == 2
    assert up.up_debug_bounds() == 0               # the normal build; libuniprefill_debug.so returns 1
    assert up.up_max_blocks(3, 1000, 64) == 1000 // 64 + 3
    nb = up.up_max_blocks(1, 32768, 64)
    a = up.up_score_workspace_bytes(1, 32768, 32, 8, 128, 64, 128, nb)
    b = up.up_score_workspace_bytes(1, 32768, 32, 8, 128, 64, 128, nb, True)
    assert 0 < a < b
    assert up.up_score_workspace_bytes(1, 32768, 32, 8, 100, 64, 128, nb) == 0     # unsupported d_k
    assert up.up_score_workspace_bytes(1, 32768, 30, 8, 128, 64, 128, nb) == 0     # Hq % Hkv != 0
    assert up.up_score_workspace_bytes(1, 32768, 32, 8, 128, 64, 48, nb) == 0      # n must divide 128
    assert up.up_compact_workspace_bytes(4, 10_000) > 0
    assert up.up_select_workspace_bytes(nb) >= 16 * nb
    assert up.up_workspace_bytes(1, 32768, 32, 8, 128, 64, 128, nb) >= max(b, up.up_compact_workspace_bytes(1, 32768),
                                                                         up.up_select_workspace_bytes(nb))


def test_host_validation_returns_before_any_launch(lib):
    import long_context_prefill_varlen_gb300 as up
    fake = ctypes.c_void_p(0x1000)     # never dereferenced: validation fails first
    null = None
    s = lib.up_score_blocks(fake, fake, fake, 1, 4096, 32, 8, 100, 64, 128, 0.088, fake, 64, fake, null, fake,
                            1 << 20, fake, null)
    assert s == up.UP_ERR_SHAPE
    s = lib.up_score_blocks(null, fake, fake, 1, 4096, 32, 8, 128, 64, 128, 0.088, fake, 64, fake, null, fake,
                            1 << 20, fake, null)
    assert s == up.UP_ERR_ARG
    s = lib.up_score_blocks(fake, fake, fake, 1, 4096, 32, 8, 128, 48, 128, 0.088, fake, 64, fake, null, fake,
                            1 << 20, fake, null)
    assert s == up.UP_ERR_SHAPE                    # G must divide the 128-key tile
    s = lib.up_score_blocks(fake, fake, fake, 1, 4096, 32, 8, 128, 64, 128, 0.088, fake, 64, fake, null, fake,
                            16, fake, null)
    assert s == up.UP_ERR_WORKSPACE
    s = lib.up_select_topp(fake, fake, fake, 1, 4096, 64, 64, 128, 128, 1.5, fake, fake, fake, null, 0, fake, null)
    assert s == up.UP_ERR_ARG                      # p outside (0, 1]
    s = lib.up_select_topp(fake, fake, fake, 1, 4096, 64, 64, 128, 128, 0.0, fake, fake, fake, null, 0, fake, null)
    assert s == up.UP_ERR_ARG
    odd = ctypes.c_void_p(0x1001)      # a token mask that is not 16-byte aligned (a view at an odd offset)
    s = lib.up_select_topp(fake, fake, fake, 1, 4096, 64, 64, 128, 128, 0.99, fake, odd, fake, null, 0, fake, null)
    assert s == up.UP_ERR_SHAPE
    s = lib.up_select_topp(fake, fake, fake, 1, 4096, 64, 64, 128, 128, 0.99, fake, fake, fake, fake, 64, fake, null)
    assert s == up.UP_ERR_WORKSPACE                # a workspace smaller than up_select_workspace_bytes
    s = lib.up_compact(fake, fake, 1, 4096, fake, 12, null, null, fake, null, null, fake, fake, fake, fake, null,
                       null, 0, 0, fake, 1 << 20, fake, null)
    assert s == up.UP_ERR_SHAPE                    # hidden size must be a multiple of 8
    s = lib.up_compact(fake, fake, 1, 4096, fake, 64, null, null, null, null, null, fake, fake, fake, fake, null,
                       null, 0, 0, fake, 1 << 20, fake, null)
    assert s == up.UP_ERR_ARG                      # hidden without out_hidden
    s = lib.up_scatter_back(fake, fake, fake, 100, 7, fake, fake, null)
    assert s == up.UP_ERR_SHAPE
    s = lib.up_seqused(fake, fake, 4, 2, 4, fake, fake, fake, null)
    assert s == up.UP_ERR_ARG                      # layer outside [0, L)
    assert lib.up_slot_mapping(fake, fake, 1, 10, null, fake, 0, 16, fake, fake, null) == up.UP_ERR_ARG
    assert up.up_status_string(up.UP_ERR_WORKSPACE).startswith("UP_ERR_WORKSPACE")


def test_binding_fails_loudly_without_the_library(tmp_path):
    import long_context_prefill_varlen_gb300 as up
    saved = up._lib
    try:
        up._lib = None
        with pytest.raises(RuntimeError):
            up.load_library(str(tmp_path / "missing.so"))
    finally:
        up._lib = saved
