"""A random-weight LLaMA-shaped decoder stack that consumes the drop step, and its FLOPs accounting.

UniPrefill ("UniPrefill: Universal Long-Context Prefill Acceleration via Block-wise Dynamic
Sparsification", arXiv 2605.06221) drops token blocks at a full-attention layer and runs every later
sublayer on the kept tokens only (section 3.4, Eq. 7); at the end of the block the dropped tokens'
old states are carried forward into the full-length stream (Eq. 8).  The saving is the cost of the
sublayers after the drop on the dropped tokens (section 3.3, "FLOPs analysis", Eqs. 9-10).

This module is the consumer of the drop step, not part of it: its layers are library code (cuBLAS
GEMMs through torch.matmul, PyTorch's varlen flash-attention forward, torch elementwise ops), with
random weights, so that the time a drop saves on a real layer stack can be measured.  The drop step
itself (score, top-p select, compaction with its metadata and drop history, Eq. 8 scatter) runs in
libuniprefill through DropStep.

Layer l (pre-norm LLaMA block, GQA, rotary positions):
    x = h + Wo . attn(rope(Wq . rms(h)), rope(Wk . rms(h)), Wv . rms(h))     causal per request
    h' = x + Wd . (silu(Wg . rms(x)) * (Wu . rms(x)))
A drop at layer l_k (the reading of Eqs. 7-10 this module takes):
  * the attention sublayer of l_k runs on the whole stream that enters l_k (it is the full-attention
    layer that supplies the scores), and its rotated Q and K are the drop step's inputs;
  * the kept tokens' x rows (H^(b,1)) are compacted, together with their positions, and the FFN of
    l_k and every later layer run on the compacted stream (Eq. 7), with rotary phases from the kept
    tokens' original positions;
  * the block of a drop ends with the stack: Eq. 8 writes the kept tokens' final states into the
    buffer that holds the stream entering l_k (H^(b,0)), so a dropped token carries the state it had
    at the input of layer l_k.  A later drop acts on the stream an earlier drop left, and the blocks
    are closed innermost first.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from .step import DropStep


@dataclass(frozen=True)
class StackGeometry:
    """Shape of one decoder layer: hidden size d, query / KV heads, head dim, FFN width."""
    d: int = 4096
    Hq: int = 32
    Hkv: int = 8
    dk: int = 128
    ffn: int = 14336
    rope_theta: float = 500000.0
    eps: float = 1e-5


LLAMA_3_1_8B = StackGeometry()


# ------------------------------------------------------------------------------------------ FLOPs accounting

def linear_flops_per_token(g: StackGeometry, attention=True, ffn=True):
    """multiply-add FLOPs (2 per MAC) of one token through one layer's projections"""
    f = 0
    if attention:
        f += 2 * g.d * (g.Hq + 2 * g.Hkv) * g.dk + 2 * g.Hq * g.dk * g.d       # Wq, Wk, Wv, Wo
    if ffn:
        f += 2 * g.d * 2 * g.ffn + 2 * g.ffn * g.d                             # Wg, Wu, Wd
    return f


def attention_flops(lengths, g: StackGeometry):
    """causal S = Q K^T and P V of every request: 2 matmuls x 2 FLOPs x Hq x dk x N(N+1)/2"""
    return sum(4 * g.Hq * g.dk * (int(N) * (int(N) + 1) // 2) for N in lengths)


def layer_flops(lengths, g: StackGeometry, attention=True, ffn=True):
    T = sum(int(N) for N in lengths)
    f = T * linear_flops_per_token(g, attention, ffn)
    if attention:
        f += attention_flops(lengths, g)
    return f


def stack_flops(lengths, g: StackGeometry, L, drops=()):
    """FLOPs of an L-layer stack over requests of the given lengths.  `drops` lists (layer, kept lengths)
    in increasing layer order: the drop layer's attention runs on the stream entering it, its FFN and
    every later layer on the kept lengths."""
    cur, total, k = list(lengths), 0, 0
    drops = list(drops)
    for layer in range(L):
        if k < len(drops) and drops[k][0] == layer:
            total += layer_flops(cur, g, ffn=False)
            cur = list(drops[k][1])
            k += 1
            total += layer_flops(cur, g, attention=False)
        else:
            total += layer_flops(cur, g)
    if k != len(drops):
        raise ValueError("drop layers must be distinct, increasing and below L")
    return total


# ------------------------------------------------------------------------------------------ the stack

def _rms(x, eps):
    xf = x.float()
    return (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + eps)).to(torch.bfloat16)


def rope_tables(positions, dk, theta):
    """cos and sin [T, dk/2] (fp32) of the rotary phases pos * theta^(-2i/dk)"""
    i = torch.arange(dk // 2, device=positions.device, dtype=torch.float32)
    inv = torch.pow(torch.tensor(theta, dtype=torch.float32, device=positions.device), -2.0 * i / dk)
    ang = positions.to(torch.float32)[:, None] * inv[None, :]
    return torch.cos(ang), torch.sin(ang)


def apply_rope(x, cos, sin):
    """rotate the pairs (j, j + dk/2) of every head of x [T, H, dk] by the token's phases"""
    h = x.shape[-1] // 2
    xf = x.float()
    x1, x2 = xf[..., :h], xf[..., h:]
    c, s = cos[:, None, :], sin[:, None, :]
    return torch.cat((x1 * c - x2 * s, x2 * c + x1 * s), dim=-1).to(torch.bfloat16).contiguous()


def varlen_causal_attention(q, k, v, cu_seqlens, max_len, scale):
    """PyTorch's flash-attention forward over a packed varlen stream (GQA: Hq a multiple of Hkv)"""
    out = torch.ops.aten._flash_attention_forward(q, k, v, cu_seqlens, cu_seqlens, int(max_len), int(max_len), 0.0,
                                                   True, False, scale=scale)
    return out[0]


class RandomLlamaStack:
    """L pre-norm decoder layers with seeded random bf16 weights (N(0, 1/fan_in); the two projections
    that feed the residual stream scaled down by sqrt(2L) so that the stream stays O(1) in bf16)."""

    def __init__(self, L, geom: StackGeometry = LLAMA_3_1_8B, seed=0, device="cuda", init_device=None):
        self.L, self.g = L, geom
        self.device = torch.device(device)
        init_device = torch.device(init_device) if init_device is not None else self.device
        gen = torch.Generator(device=init_device)
        gen.manual_seed(seed)
        g = geom

        def w(fan_in, fan_out, extra=1.0):
            t = torch.randn(fan_in, fan_out, generator=gen, device=init_device, dtype=torch.float32)
            return (t * (extra / fan_in ** 0.5)).to(torch.bfloat16).to(self.device)

        res = (2.0 * L) ** -0.5
        self.layers = []
        for _ in range(L):
            self.layers.append(dict(wq=w(g.d, g.Hq * g.dk), wk=w(g.d, g.Hkv * g.dk), wv=w(g.d, g.Hkv * g.dk),
                                    wo=w(g.Hq * g.dk, g.d, res), wgu=w(g.d, 2 * g.ffn), wd=w(g.ffn, g.d, res)))

    # one sublayer each; T = rows of the stream they are given
    def attention_sublayer(self, layer, h, positions, cu_seqlens, max_len):
        """x = h + Wo . attn(...); also returns the rotated q [T, Hq, dk] and k [T, Hkv, dk]"""
        g, Wt = self.g, self.layers[layer]
        T = h.shape[0]
        a = _rms(h, g.eps)
        cos, sin = rope_tables(positions, g.dk, g.rope_theta)
        q = apply_rope(torch.matmul(a, Wt["wq"]).view(T, g.Hq, g.dk), cos, sin)
        k = apply_rope(torch.matmul(a, Wt["wk"]).view(T, g.Hkv, g.dk), cos, sin)
        v = torch.matmul(a, Wt["wv"]).view(T, g.Hkv, g.dk)
        o = varlen_causal_attention(q, k, v, cu_seqlens, max_len, g.dk ** -0.5)
        x = h + torch.matmul(o.reshape(T, g.Hq * g.dk), Wt["wo"])
        return x, q, k

    def ffn_sublayer(self, layer, x):
        g, Wt = self.g, self.layers[layer]
        gu = torch.matmul(_rms(x, g.eps), Wt["wgu"])
        act = (torch.nn.functional.silu(gu[:, :g.ffn].float()) * gu[:, g.ffn:].float()).to(torch.bfloat16)
        return x + torch.matmul(act, Wt["wd"])

    def forward(self, hidden, positions, cu_seqlens, max_len, drops=(), upto=None, G=64, n=128, A=128,
                keep_scored=False):
        """Run layers [0, upto) (all by default) over the packed stream `hidden` [T, d] bf16 with
        `positions` [T] int64 and `cu_seqlens` [R+1] int32 (device); `max_len` bounds every request's
        length.  `drops` lists (layer, p) in increasing layer order.  Returns the full-length output
        (a new tensor; `hidden` is not written) and, per drop, a dict with its DropStep, the kept token
        count and (keep_scored) the rotated q and k it was scored on, and the stream x and positions it
        compacted.  Each drop synchronises the host
        once, to learn the compacted stream's length."""
        upto = self.L if upto is None else upto
        drops = list(drops)
        h = hidden.clone()
        pos, cu, T = positions, cu_seqlens, hidden.shape[0]
        k = 0
        stack_of_blocks = []          # (block input buffer H^(b,0), DropStep), innermost last
        info = []
        for layer in range(upto):
            x, q, kk = self.attention_sublayer(layer, h, pos, cu, max_len)
            if k < len(drops) and drops[k][0] == layer:
                p = drops[k][1]
                step = DropStep(cu, T, self.g.Hq, self.g.Hkv, self.g.dk, self.g.d, G=G, n=n, A=A, p=p, L=self.L,
                                layer=layer, device=self.device)
                step.score(q, kk)
                step.select()
                step.compact(x, pos)
                T = int(step.num_actual.item())
                step.check()
                stack_of_blocks.append((h, step))
                info.append(dict(layer=layer, p=p, step=step, kept_tokens=T,
                                 scored=(q, kk, x, pos) if keep_scored else None))
                x = step.out_hidden[:T]
                pos = step.out_positions[:T]
                cu = step.new_cu
                k += 1
            h = self.ffn_sublayer(layer, x)
        for block_in, step in reversed(stack_of_blocks):       # Eq. 8, innermost block first
            step.scatter_back(h.contiguous(), block_in)
            h = block_in
        for _, step in stack_of_blocks:
            step.check()
        return h, info
