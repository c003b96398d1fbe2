"""Device-side generation of the synthetic workloads (bit-identical to synth.cpu)."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np
import torch

from . import cpu
from .recipe import HOT_SHIFT, SINK_SCALE, SINK_TOKENS, TID_HIDDEN, TID_K, TID_Q, TID_SLOTS

_DIR = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_DIR, "csrc", "synth_gen.cu")
LIB = os.path.join(_DIR, "libupsynth.so")
_lib = None


def build(force=False):
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + ".tmp"
    cmd = [exe, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for synth_gen.cu:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB)
        vp, u64, i32, i64, f32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.synth_normal_bf16.argtypes = [vp, u64, u64, u64, vp]
        lib.synth_slots.argtypes = [vp, u64, u64, u64, vp]
        lib.synth_positions.argtypes = [vp, vp, i32, i64, vp]
        lib.synth_plant_k.argtypes = [vp, vp, i32, i64, i32, i32, vp, vp, i32, f32, f32, vp]
        for f in (lib.synth_normal_bf16, lib.synth_slots, lib.synth_positions, lib.synth_plant_k):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ok(code, what):
    if code != 0:
        raise RuntimeError(f"{what}: CUDA error {code}")


def normal_bf16(key, start, count, device="cuda"):
    out = torch.empty(count, dtype=torch.bfloat16, device=device)
    _ok(_load().synth_normal_bf16(ctypes.c_void_p(out.data_ptr()), key, start, count, _s()), "synth_normal_bf16")
    return out


def build_device(w, device="cuda", parts=("Q", "K", "hidden", "positions", "slots"), u=None, hot_tok=None):
    """Every input of one drop step generated in device memory; u and the hot mask come from the host."""
    lib = _load()
    out = {}
    cu = torch.tensor(w.cu_seqlens(), dtype=torch.int32, device=device)
    out["cu_seqlens"] = cu
    T = w.T
    if "Q" in parts:
        out["Q"] = normal_bf16(w.key(TID_Q), 0, T * w.Hq * w.dk, device).view(T, w.Hq, w.dk)
    if "K" in parts:
        K = normal_bf16(w.key(TID_K), 0, T * w.Hkv * w.dk, device).view(T, w.Hkv, w.dk)
        u = cpu.mean_query_dirs(w) if u is None else u
        hot_tok = cpu.hot_token_mask(w) if hot_tok is None else hot_tok
        ud = torch.from_numpy(np.ascontiguousarray(u)).to(device)
        hd = torch.from_numpy(np.ascontiguousarray(hot_tok)).to(device)
        _ok(lib.synth_plant_k(ctypes.c_void_p(K.data_ptr()), ctypes.c_void_p(cu.data_ptr()), w.R, T, w.Hkv, w.dk,
                              ctypes.c_void_p(hd.data_ptr()), ctypes.c_void_p(ud.data_ptr()), SINK_TOKENS,
                              SINK_SCALE, HOT_SHIFT, _s()), "synth_plant_k")
        out["K"] = K
        out["u"], out["hot_tok"] = u, hot_tok
    if "hidden" in parts:
        out["hidden"] = normal_bf16(w.key(TID_HIDDEN), 0, T * w.hdim, device).view(T, w.hdim)
    if "positions" in parts:
        pos = torch.empty(max(1, T), dtype=torch.int64, device=device)[:T]
        _ok(lib.synth_positions(ctypes.c_void_p(pos.data_ptr()), ctypes.c_void_p(cu.data_ptr()), w.R, T, _s()),
            "synth_positions")
        out["positions"] = pos
    if "slots" in parts:
        sl = torch.empty(max(1, T), dtype=torch.int64, device=device)[:T]
        _ok(lib.synth_slots(ctypes.c_void_p(sl.data_ptr()), w.key(TID_SLOTS), 0, T, _s()), "synth_slots")
        out["slots"] = sl
    return out


def to_device(host, device="cuda"):
    """Upload numpy inputs from synth.cpu.materialize (small workloads)."""
    d = {}
    for k, v in host.items():
        if isinstance(v, np.ndarray):
            t = torch.from_numpy(np.ascontiguousarray(v))
            if v.dtype == np.uint16:
                t = t.view(torch.bfloat16)
            d[k] = t.to(device)
        else:
            d[k] = v
    d["cu_seqlens"] = d["cu_seqlens"].to(torch.int32)
    return d
