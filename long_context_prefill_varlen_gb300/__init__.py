"""Python binding of libuniprefill.so: UniPrefill's per-layer token-dropping hot path on GB300.

Each ``up_*`` function has the name and meaning of the C entry point declared in
include/uniprefill.h and does argument marshalling only (torch tensors -> device
pointers, sizes, the current CUDA stream); every step of the computation runs in
the library's CUDA kernels.  There is no CPU fallback: if the shared library is
missing or cannot be loaded, importing the binding's functions raises.

Paper: "UniPrefill: Universal Long-Context Prefill Acceleration via Block-wise
Dynamic Sparsification" (arXiv 2605.06221), sections 3.2-3.5.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libuniprefill.so")

UP_OK, UP_ERR_ARG, UP_ERR_SHAPE, UP_ERR_WORKSPACE, UP_ERR_CUDA, UP_ERR_DEVICE = range(6)
MAX_BLOCKS_PER_REQUEST = 8192
NOALLOC_MAX_TOKENS = 16384 * 1024

_c_p = ctypes.c_void_p
_i32, _i64, _f32, _f64, _sz, _u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_size_t, ctypes.c_uint64

_SIGNATURES = {
    "up_max_blocks": (_i64, [_i32, _i64, _i32]),
    "up_score_workspace_bytes": (_sz, [_i32, _i64, _i32, _i32, _i32, _i32, _i32, _i64, _i32]),
    "up_compact_workspace_bytes": (_sz, [_i32, _i64]),
    "up_select_workspace_bytes": (_sz, [_i64]),
    "up_workspace_bytes": (_sz, [_i32, _i64, _i32, _i32, _i32, _i32, _i32, _i64]),
    "up_make_cu_blocks": (_i32, [_c_p, _i32, _i64, _i32, _c_p, _c_p, _c_p]),
    "up_score_blocks": (_i32, [_c_p, _c_p, _c_p, _i32, _i64, _i32, _i32, _i32, _i32, _i32, _f32,
                                _c_p, _i64, _c_p, _c_p, _c_p, _sz, _c_p, _c_p]),
    "up_select_topp": (_i32, [_c_p, _c_p, _c_p, _i32, _i64, _i64, _i32, _i32, _i32, _f64,
                               _c_p, _c_p, _c_p, _c_p, _sz, _c_p, _c_p]),
    "up_compact": (_i32, [_c_p, _c_p, _i32, _i64, _c_p, _i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                           _c_p, _c_p, _c_p, _c_p, _c_p, _i32, _i32, _c_p, _sz, _c_p, _c_p]),
    "up_compact_noalloc": (_i32, [_c_p, _c_p, _i32, _i64, _c_p, _i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                                   _c_p, _c_p, _c_p, _c_p, _c_p, _i32, _i32, _c_p, _c_p]),
    "up_scatter_back": (_i32, [_c_p, _c_p, _c_p, _i64, _i32, _c_p, _c_p, _c_p]),
    "up_slot_mapping": (_i32, [_c_p, _c_p, _i32, _i64, _c_p, _c_p, _i32, _i32, _c_p, _c_p, _c_p]),
    "up_seqused": (_i32, [_c_p, _c_p, _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p]),
    "up_read_status": (_i32, [_c_p, _c_p, _c_p]),
    "up_status_string": (ctypes.c_char_p, [_i32, _i32]),
    "up_kernel_launches": (_u64, []),
    "up_abi_version": (_i32, []),
    "up_debug_bounds": (_i32, []),
}

_lib = None


def load_library(path=LIB_PATH):
    """Load libuniprefill.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libuniprefill.so not found at {path}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class UpError(RuntimeError):
    def __init__(self, code, where):
        msg = load_library().up_status_string(code, 0).decode()
        super().__init__(f"{where}: {msg}")
        self.code = code


def _check(code, where):
    if code != UP_OK:
        raise UpError(code, where)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _bf16(t):
    assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.is_cuda
    return _p(t)


# ------------------------------------------------------------------------------------------ sizing

def up_max_blocks(R, T, G):
    return load_library().up_max_blocks(R, T, G)


def up_score_workspace_bytes(R, T, Hq, Hkv, dk, G, n, nb_cap, with_token_scores=False):
    return load_library().up_score_workspace_bytes(R, T, Hq, Hkv, dk, G, n, nb_cap, int(bool(with_token_scores)))


def up_compact_workspace_bytes(R, T):
    return load_library().up_compact_workspace_bytes(R, T)


def up_select_workspace_bytes(nb_cap):
    return load_library().up_select_workspace_bytes(nb_cap)


def up_workspace_bytes(R, T, Hq, Hkv, dk, G, n, nb_cap):
    return load_library().up_workspace_bytes(R, T, Hq, Hkv, dk, G, n, nb_cap)


# ------------------------------------------------------------------------------------------ the drop step

def up_make_cu_blocks(cu_seqlens, G, cu_blocks, dev_status, T=None, stream=None):
    R = cu_seqlens.numel() - 1
    T = int(T) if T is not None else None
    if T is None:
        raise ValueError("T (total tokens) is required: the binding never reads device memory back")
    _check(load_library().up_make_cu_blocks(_p(cu_seqlens), R, T, G, _p(cu_blocks), _p(dev_status), _stream(stream)),
           "up_make_cu_blocks")


def up_score_blocks(Q, K, cu_seqlens, G, n, cu_blocks, block_scores, ws, dev_status, token_scores=None,
                    sm_scale=None, stream=None):
    T, Hq, dk = Q.shape
    Hkv = K.shape[1]
    R = cu_seqlens.numel() - 1
    sm_scale = dk ** -0.5 if sm_scale is None else sm_scale
    _check(load_library().up_score_blocks(_bf16(Q), _bf16(K), _p(cu_seqlens), R, T, Hq, Hkv, dk, G, n, sm_scale,
                                          _p(cu_blocks), block_scores.numel(), _p(block_scores), _p(token_scores),
                                          _p(ws), ws.numel() * ws.element_size(), _p(dev_status), _stream(stream)),
           "up_score_blocks")


def up_select_topp(block_scores, cu_blocks, cu_seqlens, T, G, n, A, p, block_keep, token_keep, kstar, dev_status,
                   ws=None, stream=None):
    """ws: optional device workspace (up_select_workspace_bytes(block_scores.numel()) bytes); needed only
    for requests of more than MAX_BLOCKS_PER_REQUEST blocks."""
    R = cu_seqlens.numel() - 1
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load_library().up_select_topp(_p(block_scores), _p(cu_blocks), _p(cu_seqlens), R, T, block_scores.numel(),
                                         G, n, A, float(p), _p(block_keep), _p(token_keep), _p(kstar), _p(ws), nbytes,
                                         _p(dev_status), _stream(stream)),
           "up_select_topp")


def up_compact(token_keep, cu_seqlens, kept_index, new_cu_seqlens, new_seq_lens, num_actual_tokens, ws, dev_status,
               hidden=None, out_hidden=None, positions=None, out_positions=None, slots=None, out_slots=None,
               kept_len=None, drop_layer=None, layer=0, stream=None):
    R = cu_seqlens.numel() - 1
    T = token_keep.numel()
    hdim = hidden.shape[1] if hidden is not None else 0
    L = drop_layer.numel() if drop_layer is not None else (kept_len.shape[0] if kept_len is not None else 0)
    _check(load_library().up_compact(_p(token_keep), _p(cu_seqlens), R, T, _p(hidden), hdim, _p(positions), _p(slots),
                                     _p(out_hidden), _p(out_positions), _p(out_slots), _p(kept_index),
                                     _p(new_cu_seqlens), _p(new_seq_lens), _p(num_actual_tokens), _p(kept_len),
                                     _p(drop_layer), L, layer, _p(ws), ws.numel() * ws.element_size(),
                                     _p(dev_status), _stream(stream)),
           "up_compact")


def up_compact_noalloc(token_keep, cu_seqlens, kept_index, new_cu_seqlens, new_seq_lens, num_actual_tokens,
                       dev_status, hidden=None, out_hidden=None, positions=None, out_positions=None, slots=None,
                       out_slots=None, kept_len=None, drop_layer=None, layer=0, stream=None):
    """up_compact for callers that cannot provide a device workspace: the library's own fixed scratch
    array is used instead (at most UP_NOALLOC_MAX_TOKENS tokens; calls that overlap on the GPU race)."""
    R = cu_seqlens.numel() - 1
    T = token_keep.numel()
    hdim = hidden.shape[1] if hidden is not None else 0
    L = drop_layer.numel() if drop_layer is not None else (kept_len.shape[0] if kept_len is not None else 0)
    _check(load_library().up_compact_noalloc(_p(token_keep), _p(cu_seqlens), R, T, _p(hidden), hdim, _p(positions),
                                             _p(slots), _p(out_hidden), _p(out_positions), _p(out_slots),
                                             _p(kept_index), _p(new_cu_seqlens), _p(new_seq_lens),
                                             _p(num_actual_tokens), _p(kept_len), _p(drop_layer), L, layer,
                                             _p(dev_status), _stream(stream)),
           "up_compact_noalloc")


def up_scatter_back(new_states, kept_index, num_actual_tokens, residual, dev_status, stream=None):
    """residual [T, hdim] receives the compacted rows new_states [T_upper <= T, hdim] (T_upper is
    passed as the bound of *num_actual_tokens)."""
    T, hdim = residual.shape
    assert new_states.shape[1] == hdim and new_states.shape[0] <= T
    _check(load_library().up_scatter_back(_bf16(new_states), _p(kept_index), _p(num_actual_tokens),
                                          new_states.shape[0], hdim, _bf16(residual), _p(dev_status),
                                          _stream(stream)),
           "up_scatter_back")


def up_slot_mapping(positions, cu_seqlens, block_table, B, slots, dev_status, num_tokens=None, stream=None):
    R = cu_seqlens.numel() - 1
    _check(load_library().up_slot_mapping(_p(positions), _p(cu_seqlens), R, positions.numel(), _p(num_tokens),
                                          _p(block_table), block_table.shape[1], B, _p(slots), _p(dev_status),
                                          _stream(stream)),
           "up_slot_mapping")


def up_seqused(kept_len, drop_layer, layer, orig_len, kv_len, seqused, stream=None):
    L, R = kept_len.shape
    _check(load_library().up_seqused(_p(kept_len), _p(drop_layer), L, R, layer, _p(orig_len), _p(kv_len),
                                     _p(seqused), _stream(stream)),
           "up_seqused")


def up_read_status(dev_status, stream=None):
    out = ctypes.c_int32(0)
    code = load_library().up_read_status(_p(dev_status), ctypes.byref(out), _stream(stream))
    if code not in (UP_OK, UP_ERR_DEVICE):
        _check(code, "up_read_status")
    return out.value


def up_status_string(code, device=False):
    return load_library().up_status_string(code, int(bool(device))).decode()


def up_kernel_launches():
    return int(load_library().up_kernel_launches())


def up_abi_version():
    return int(load_library().up_abi_version())


def up_debug_bounds():
    return int(load_library().up_debug_bounds())


from .step import DropStep  # noqa: E402,F401
