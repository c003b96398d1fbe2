"""Float64 CPU recomputation of the random-weight decoder stack (test infrastructure).

Plain formulas, one request and one head at a time: pre-norm RMS normalisation, rotary phases on the
pairs (j, j + dk/2), causal softmax attention with GQA head sharing, SwiGLU FFN.  Drops follow the
reading of UniPrefill section 3.4 (Eqs. 7-8) that the stack takes: the drop layer's attention runs on
the stream entering it, the kept rows of its output continue through the FFN and every later layer,
and at the end each block's input buffer receives its kept rows' final states, innermost block first.
The keep masks are inputs (the decision itself is the operator's, checked against the oracle
elsewhere).

`rowwise=True` computes each query row's causal scores against exactly the keys it sees (for FLOP
counting: S and P V then cost 2 * dk per visible key and head).
"""
from __future__ import annotations

import numpy as np
import torch


def _w(stack, layer, name):
    return stack.layers[layer][name].detach().to("cpu", torch.float64)


def _rms(x, eps):
    return x / torch.sqrt((x * x).mean(-1, keepdim=True) + eps)


def _rope(x, positions, dk, theta):
    """x [T, H, dk] float64; phases pos * theta^(-2i/dk) computed in float32 like the stack's tables"""
    i = torch.arange(dk // 2, dtype=torch.float32)
    inv = torch.pow(torch.tensor(theta, dtype=torch.float32), -2.0 * i / dk)
    ang = (torch.as_tensor(positions).to(torch.float32)[:, None] * inv[None, :]).to(torch.float64)
    c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    h = dk // 2
    x1, x2 = x[..., :h], x[..., h:]
    return torch.cat((x1 * c - x2 * s, x2 * c + x1 * s), dim=-1)


def _attention(q, k, v, lengths, scale, group, rowwise):
    T, Hq, dk = q.shape
    out = torch.zeros_like(q)
    start = 0
    for N in lengths:
        N = int(N)
        for hq in range(Hq):
            hk = hq // group
            qs, ks, vs = q[start:start + N, hq], k[start:start + N, hk], v[start:start + N, hk]
            if rowwise:
                for i in range(N):                       # 1-row matrix products (counted as mm)
                    s = torch.matmul(qs[i:i + 1], ks[:i + 1].T) * scale
                    p = torch.softmax(s, dim=1)
                    out[start + i, hq] = torch.matmul(p, vs[:i + 1])[0]
            elif N:
                s = torch.matmul(qs, ks.T) * scale
                s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
                out[start:start + N, hq] = torch.matmul(torch.softmax(s, dim=1), vs)
        start += N
    return out


def attention_sublayer(stack, layer, h, positions, lengths, rowwise=False):
    g = stack.g
    T = h.shape[0]
    a = _rms(h, g.eps)
    q = _rope(torch.matmul(a, _w(stack, layer, "wq")).view(T, g.Hq, g.dk), positions, g.dk, g.rope_theta)
    k = _rope(torch.matmul(a, _w(stack, layer, "wk")).view(T, g.Hkv, g.dk), positions, g.dk, g.rope_theta)
    v = torch.matmul(a, _w(stack, layer, "wv")).view(T, g.Hkv, g.dk)
    o = _attention(q, k, v, lengths, g.dk ** -0.5, g.Hq // g.Hkv, rowwise)
    return h + torch.matmul(o.reshape(T, g.Hq * g.dk), _w(stack, layer, "wo"))


def ffn_sublayer(stack, layer, x):
    g = stack.g
    gu = torch.matmul(_rms(x, g.eps), _w(stack, layer, "wgu"))
    act = torch.nn.functional.silu(gu[:, :g.ffn]) * gu[:, g.ffn:]
    return x + torch.matmul(act, _w(stack, layer, "wd"))


def forward(stack, hidden, positions, lengths, drops=(), upto=None, rowwise=False):
    """hidden [T, d] (any float dtype), positions [T] int, lengths per request; drops = [(layer, keep)]
    with keep a bool array over the stream entering that layer.  Returns the float64 output [T, d]."""
    upto = stack.L if upto is None else upto
    h = torch.as_tensor(hidden).to("cpu", torch.float64)
    pos = np.asarray(positions)
    lengths = [int(N) for N in lengths]
    drops = list(drops)
    blocks, k = [], 0
    for layer in range(upto):
        x = attention_sublayer(stack, layer, h, pos, lengths, rowwise)
        if k < len(drops) and drops[k][0] == layer:
            keep = np.asarray(drops[k][1], dtype=bool)
            assert keep.size == h.shape[0]
            blocks.append((h, keep))
            cu = np.concatenate([[0], np.cumsum(lengths)])
            lengths = [int(keep[cu[r]:cu[r + 1]].sum()) for r in range(len(lengths))]
            x = x[torch.from_numpy(keep)]
            pos = pos[keep]
            k += 1
        h = ffn_sublayer(stack, layer, x)
    for block_in, keep in reversed(blocks):
        full = block_in.clone()
        full[torch.from_numpy(keep)] = h
        h = full
    return h
