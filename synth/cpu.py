"""numpy implementation of the counter-based input generator.

Definitions (the CUDA twin in synth/csrc/synth_gen.cu implements the same):

* ``mix64`` is the output function of splitmix64 (Steele, Lea & Flood 2014):
  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
  z ^= z >> 31 (all modulo 2**64).
* ``stream_key(seed, tid) = mix64(mix64(seed + GAMMA) + tid * GAMMA)``.
* word ``k`` of element ``idx`` of a stream is the (3*idx + k + 1)-th splitmix64
  output from state ``key``: ``mix64(key + (3*idx + k + 1) * GAMMA)``.
* N(0,1)-like value: Irwin-Hall sum of twelve 16-bit uniforms (the four 16-bit
  fields of words 0, 1, 2): ``z = (S - 393210) * 2**-16`` (exact in fp32,
  variance 12 * (65536**2 - 1) / 12 / 2**32 ~= 1), rounded to bf16 with
  round-to-nearest-even on the fp32 bit pattern.
* uniform in [0, 1): ``(word0 >> 11) * 2**-53``.
"""
from __future__ import annotations

import math
import os

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1
IH_OFFSET = 6 * 65535            # mean of the twelve-term sum
_CHUNK = 1 << 18


def _mix64_int(z):
    z &= M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def stream_key(seed, tid):
    return _mix64_int((_mix64_int(seed + GAMMA) + tid * GAMMA) & M64)


def mix64(z):
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def _word(key, idx, k):
    ctr = idx * np.uint64(3) + np.uint64(k + 1)
    return mix64(np.uint64(key) + ctr * np.uint64(GAMMA))


def f32_to_bf16_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bit pattern (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_chunk(key, start, count):
    lanes = np.uint64(0x0000FFFF0000FFFF)
    idx = np.arange(start, start + count, dtype=np.uint64)
    acc = np.zeros(count, dtype=np.uint64)
    for k in range(3):
        w = _word(key, idx, k)
        # two 32-bit lanes, each the sum of two 16-bit fields (no carry across lanes)
        acc += (w & lanes) + ((w >> np.uint64(16)) & lanes)
    s = (acc & np.uint64(0xFFFFFFFF)) + (acc >> np.uint64(32))
    z = (s.astype(np.int64) - IH_OFFSET).astype(np.float32) * np.float32(2.0 ** -16)
    return f32_to_bf16_bits(z)


def normal_bf16_bits(key, start, count):
    """bf16 bit patterns of elements [start, start+count) of stream ``key``."""
    out = np.empty(count, dtype=np.uint16)
    spans = [(c0, min(count, c0 + _CHUNK)) for c0 in range(0, count, _CHUNK)]

    def run(span):
        c0, c1 = span
        with np.errstate(over="ignore"):
            out[c0:c1] = _normal_chunk(key, start + c0, c1 - c0)

    if len(spans) > 2:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(run, spans))
    else:
        for sp in spans:
            run(sp)
    return out


def uniform01(key, start, count):
    with np.errstate(over="ignore"):
        idx = np.arange(start, start + count, dtype=np.uint64)
        w = _word(key, idx, 0)
    return (w >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def slot_values(key, start, count):
    """Opaque int64 KV-slot ids (40-bit) for the tokens [start, start+count)."""
    with np.errstate(over="ignore"):
        idx = np.arange(start, start + count, dtype=np.uint64)
        w = _word(key, idx, 0)
    return (w & np.uint64((1 << 40) - 1)).astype(np.int64)


# --------------------------------------------------------------------------------------
# planted structure


def hot_blocks(w):
    """Per request: sorted list of hot block indices (never a sink or window block)."""
    from .recipe import TID_HOTFRAC, TID_HOTPICK
    kf = w.key(TID_HOTFRAC)
    kp = w.key(TID_HOTPICK)
    out = []
    for r, N in enumerate(w.lengths):
        nb = -(-N // w.G)
        elig = [g for g in range(nb) if g * w.G >= w.A and (g + 1) * w.G <= N - w.n]
        kind = w.hot[0]
        if kind == "count":
            cnt = int(w.hot[1])
        elif kind == "frac":
            cnt = int(math.ceil(w.hot[1] * nb))
        elif kind == "uniform":
            f = w.hot[1] + (w.hot[2] - w.hot[1]) * float(uniform01(kf, r, 1)[0])
            cnt = int(math.ceil(f * nb))
        else:
            raise ValueError(kind)
        cnt = max(0, min(cnt, len(elig)))
        u = uniform01(kp, r << 24, max(cnt, 1))
        for i in range(cnt):  # partial Fisher-Yates
            j = i + int(math.floor(float(u[i]) * (len(elig) - i)))
            elig[i], elig[j] = elig[j], elig[i]
        out.append(sorted(elig[:cnt]))
    return out


def hot_token_mask(w, hot=None):
    hot = hot_blocks(w) if hot is None else hot
    cu = w.cu_seqlens()
    m = np.zeros(w.T, dtype=np.uint8)
    for r, blocks in enumerate(hot):
        N = w.lengths[r]
        for g in blocks:
            m[cu[r] + g * w.G: cu[r] + min(N, (g + 1) * w.G)] = 1
    return m


def gen_q(w, t0, t1):
    """Q bf16 bits [t1-t0, Hq, dk] for packed tokens [t0, t1)."""
    from .recipe import TID_Q
    e = w.Hq * w.dk
    return normal_bf16_bits(w.key(TID_Q), t0 * e, (t1 - t0) * e).reshape(t1 - t0, w.Hq, w.dk)


def window_tokens(w, r):
    cu = w.cu_seqlens()
    N = w.lengths[r]
    ne = min(w.n, N)
    return cu[r] + N - ne, cu[r] + N


def mean_query_dirs(w):
    """u[r, kh, :]: unit vector of the fp64 mean of the group's window query rows, fp32."""
    u = np.zeros((w.R, w.Hkv, w.dk), dtype=np.float32)
    for r in range(w.R):
        a, b = window_tokens(w, r)
        if b <= a:
            continue
        q = bf16_bits_to_f32(gen_q(w, a, b)).astype(np.float64)
        for kh in range(w.Hkv):
            m = q[:, kh * w.group:(kh + 1) * w.group, :].reshape(-1, w.dk).mean(axis=0)
            nrm = math.sqrt(float((m * m).sum()))
            if nrm > 0:
                u[r, kh] = (m / nrm).astype(np.float32)
    return u


def token_request(w, t0, t1):
    cu = np.asarray(w.cu_seqlens(), dtype=np.int64)
    t = np.arange(t0, t1, dtype=np.int64)
    r = np.searchsorted(cu, t, side="right") - 1
    return r, t - cu[r]


def gen_k(w, t0, t1, u=None, hot_tok=None):
    """K bf16 bits [t1-t0, Hkv, dk] with the sink scale and the hot shift applied."""
    from .recipe import TID_K, SINK_TOKENS, SINK_SCALE, HOT_SHIFT
    e = w.Hkv * w.dk
    k = normal_bf16_bits(w.key(TID_K), t0 * e, (t1 - t0) * e).reshape(t1 - t0, w.Hkv, w.dk)
    u = mean_query_dirs(w) if u is None else u
    hot_tok = hot_token_mask(w) if hot_tok is None else hot_tok
    req, loc = token_request(w, t0, t1)
    sink = loc < SINK_TOKENS
    if sink.any():
        k[sink] = f32_to_bf16_bits(bf16_bits_to_f32(k[sink]) * np.float32(SINK_SCALE))
    hot = hot_tok[t0:t1].astype(bool)
    if hot.any():
        kf = bf16_bits_to_f32(k[hot])
        shift = np.float32(HOT_SHIFT) * u[req[hot]]          # exact (power of two)
        k[hot] = f32_to_bf16_bits(kf + shift)                # one fp32 rounding, then RNE to bf16
    return k


def gen_hidden(w, t0, t1):
    from .recipe import TID_HIDDEN
    return normal_bf16_bits(w.key(TID_HIDDEN), t0 * w.hdim, (t1 - t0) * w.hdim).reshape(t1 - t0, w.hdim)


def gen_positions(w, t0=0, t1=None):
    t1 = w.T if t1 is None else t1
    return token_request(w, t0, t1)[1].astype(np.int64)


def gen_slots(w, t0=0, t1=None):
    from .recipe import TID_SLOTS
    t1 = w.T if t1 is None else t1
    return slot_values(w.key(TID_SLOTS), t0, t1 - t0)


def materialize(w, with_hidden=True):
    """Every input of one drop step on the host (small workloads only)."""
    u = mean_query_dirs(w)
    hot = hot_blocks(w)
    hot_tok = hot_token_mask(w, hot)
    d = dict(
        cu_seqlens=np.asarray(w.cu_seqlens(), dtype=np.int32),
        Q=gen_q(w, 0, w.T), K=gen_k(w, 0, w.T, u, hot_tok), u=u, hot=hot, hot_tok=hot_tok,
        positions=gen_positions(w), slots=gen_slots(w))
    if with_hidden:
        d["hidden"] = gen_hidden(w, 0, w.T)
    return d
