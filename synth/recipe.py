"""Workload recipes: the shapes of the paper's evaluation settings, synthetic.

The paper (UniPrefill: Universal Long-Context Prefill Acceleration via
Block-wise Dynamic Sparsification, arXiv 2605.06221) evaluates on RULER
prompts of 4K-128K tokens with LLaMA-3.1-8B-Instruct, Qwen3-Next-80B-A3B and
Gemma-3-12B (section 4.1; Tables 1-2), with G=64, n=128, A=128 and
p=0.99/0.99/0.98.  No dataset or weights are used here: each recipe keeps the
geometry of one full-attention layer (heads, head dim, hidden size), the
request-length mix and the hyper-parameters, and fills the tensors with
seeded N(0,1)-like bf16 values plus planted structure (hot blocks whose keys
are shifted towards the mean window query, and a 4-token attention sink).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

from . import cpu as _cpu

# tensor ids (salted by the config index so configs draw independent streams)
TID_Q, TID_K, TID_HIDDEN, TID_SLOTS, TID_LENGTHS, TID_HOTFRAC, TID_HOTPICK, TID_MISC = range(1, 9)

SINK_TOKENS = 4        # keys of the first tokens of each request are scaled
SINK_SCALE = 4.0
HOT_SHIFT = 2.0        # hot keys: K <- K + 2.0 * u (u: unit mean window query of the group)


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    lengths: tuple
    Hq: int
    Hkv: int
    dk: int
    hdim: int
    G: int
    n: int
    A: int
    p: float
    hot: tuple               # ("count", k) | ("frac", f) | ("uniform", lo, hi)
    seed: int = 0
    salt: int = field(default=None)

    @property
    def R(self):
        return len(self.lengths)

    @property
    def T(self):
        return int(sum(self.lengths))

    @property
    def group(self):
        return self.Hq // self.Hkv

    @property
    def tid_salt(self):
        return (self.index if self.salt is None else self.salt) * 16

    def key(self, tid):
        return _cpu.stream_key(self.seed, self.tid_salt + tid)

    def cu_seqlens(self):
        cu = [0]
        for L in self.lengths:
            cu.append(cu[-1] + int(L))
        return cu

    def replace(self, **kw):
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def loguniform_lengths(seed, salt, R, lo, hi):
    """R integer lengths, log-uniform in [lo, hi], from the counter stream."""
    key = _cpu.stream_key(seed, salt + TID_LENGTHS)
    u = _cpu.uniform01(key, 0, R)
    out = []
    for x in u:
        v = lo * math.exp(float(x) * math.log(hi / lo))
        out.append(int(min(hi, max(lo, math.floor(v + 0.5)))))
    return tuple(out)


def _cfg3_lengths():
    return loguniform_lengths(0, 3 * 16, 16, 4096, 131072)


CONFIGS = {
    1: Workload(1, "single request N=4096, LLaMA-3.1-8B layer geometry (32/8 heads, d_k=128, hidden 4096)",
                (4096,), 32, 8, 128, 4096, 64, 128, 128, 0.99, ("count", 8)),
    2: Workload(2, "LLaMA-3.1-8B full-attention layer, single request N=32768",
                (32768,), 32, 8, 128, 4096, 64, 128, 128, 0.99, ("frac", 0.05)),
    3: Workload(3, "continuous-batch varlen: 16 requests log-uniform in [4096, 131072], LLaMA-3.1-8B geometry",
                _cfg3_lengths(), 32, 8, 128, 4096, 64, 128, 128, 0.99, ("uniform", 0.01, 0.20)),
    4: Workload(4, "Qwen3-Next-80B-A3B full-attention layer geometry, 4 x N=131072, G=32",
                (131072,) * 4, 16, 2, 256, 2048, 32, 128, 128, 0.99, ("frac", 0.02)),
    5: Workload(5, "Gemma-3-12B full-attention layer geometry under load, 64 x N=32768",
                (32768,) * 64, 16, 8, 256, 3840, 64, 128, 128, 0.99, ("uniform", 0.01, 0.30)),
}


def workload(i, **overrides):
    w = CONFIGS[i]
    return w.replace(**overrides) if overrides else w


def small(name="small", lengths=(1000, 3000, 200, 77), Hq=8, Hkv=2, dk=128, hdim=256,
          G=64, n=128, A=128, p=0.99, hot=("frac", 0.08), seed=0, salt=17):
    """A small varlen case for parity tests: several tiles, ragged tails."""
    return Workload(0, name, tuple(lengths), Hq, Hkv, dk, hdim, G, n, A, p, hot, seed, salt)
