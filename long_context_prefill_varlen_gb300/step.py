"""DropStep: the buffers of one drop step, allocated once, and the C-ABI calls in order.

score (Eqs. 2-4) -> select (Eq. 5/14 + sinks/window) -> compact (+ metadata, drop history)
-> [the caller's sublayers run on the compacted stream, Eq. 7] -> scatter back (Eq. 8)
-> seqused (Eq. 17) for a later layer.  Only marshalling happens here; all arithmetic is
in libuniprefill's kernels.
"""
from __future__ import annotations

import torch

from . import (up_compact, up_compact_workspace_bytes, up_make_cu_blocks, up_max_blocks, up_read_status,
               up_scatter_back, up_score_blocks, up_score_workspace_bytes, up_select_topp, up_select_workspace_bytes,
               up_seqused)


class DropStep:
    def __init__(self, cu_seqlens, T, Hq, Hkv, dk, hdim, G=64, n=128, A=128, p=0.99, L=1, layer=0,
                 with_token_scores=False, device="cuda"):
        dev = torch.device(device)
        self.cu = cu_seqlens.to(device=dev, dtype=torch.int32).contiguous()
        self.R = self.cu.numel() - 1
        self.T, self.Hq, self.Hkv, self.dk, self.hdim = int(T), Hq, Hkv, dk, hdim
        self.G, self.n, self.A, self.p, self.L, self.layer = G, n, A, p, L, layer
        R, T = self.R, self.T
        self.nb_cap = up_max_blocks(R, T, G)
        i32 = dict(device=dev, dtype=torch.int32)
        self.status = torch.zeros(1, **i32)
        self.cu_blocks = torch.zeros(R + 1, **i32)
        self.block_scores = torch.zeros(max(1, self.nb_cap), device=dev, dtype=torch.float32)
        self.token_scores = torch.zeros(T, device=dev, dtype=torch.float32) if with_token_scores else None
        self.block_keep = torch.zeros(max(1, self.nb_cap), device=dev, dtype=torch.uint8)
        self.token_keep = torch.zeros(max(16, T), device=dev, dtype=torch.uint8)[:T]
        self.kstar = torch.zeros(R, **i32)
        self.kept_index = torch.zeros(max(1, T), **i32)
        self.new_cu = torch.zeros(R + 1, **i32)
        self.new_len = torch.zeros(R, **i32)
        self.num_actual = torch.zeros(1, **i32)
        self.out_hidden = torch.empty(T, hdim, device=dev, dtype=torch.bfloat16) if hdim else None
        self.out_positions = torch.empty(max(1, T), device=dev, dtype=torch.int64)
        self.out_slots = torch.empty(max(1, T), device=dev, dtype=torch.int64)
        self.kept_len = torch.zeros(L, R, **i32)
        self.drop_layer = torch.zeros(L, device=dev, dtype=torch.uint8)
        self.seqused_out = torch.zeros(R, **i32)
        sws = up_score_workspace_bytes(R, T, Hq, Hkv, dk, G, n, self.nb_cap, with_token_scores)
        if sws == 0:
            raise ValueError("unsupported geometry for up_score_blocks")
        # one workspace for the calls of the step, which run one after another on a stream
        ws = max(sws, up_compact_workspace_bytes(R, T), up_select_workspace_bytes(self.nb_cap))
        self.ws = torch.empty(ws, device=dev, dtype=torch.uint8)
        up_make_cu_blocks(self.cu, G, self.cu_blocks, self.status, T=T)

    def score(self, Q, K, stream=None):
        up_score_blocks(Q, K, self.cu, self.G, self.n, self.cu_blocks, self.block_scores, self.ws, self.status,
                        token_scores=self.token_scores, stream=stream)

    def select(self, stream=None):
        up_select_topp(self.block_scores, self.cu_blocks, self.cu, self.T, self.G, self.n, self.A, self.p,
                       self.block_keep, self.token_keep, self.kstar, self.status, ws=self.ws, stream=stream)

    def compact(self, hidden=None, positions=None, slots=None, stream=None):
        up_compact(self.token_keep, self.cu, self.kept_index, self.new_cu, self.new_len, self.num_actual, self.ws,
                   self.status, hidden=hidden, out_hidden=self.out_hidden if hidden is not None else None,
                   positions=positions, out_positions=self.out_positions[:self.T] if positions is not None else None,
                   slots=slots, out_slots=self.out_slots[:self.T] if slots is not None else None,
                   kept_len=self.kept_len, drop_layer=self.drop_layer, layer=self.layer, stream=stream)

    def scatter_back(self, new_states, residual, stream=None):
        up_scatter_back(new_states, self.kept_index, self.num_actual, residual, self.status, stream=stream)

    def seqused(self, orig_len, kv_len, layer, stream=None):
        up_seqused(self.kept_len, self.drop_layer, layer, orig_len, kv_len, self.seqused_out, stream=stream)
        return self.seqused_out

    def run(self, Q, K, hidden=None, positions=None, slots=None, residual=None, stream=None):
        """score -> select -> compact (-> scatter of the compacted rows into `residual`)."""
        self.score(Q, K, stream)
        self.select(stream)
        self.compact(hidden, positions, slots, stream)
        if residual is not None and hidden is not None:
            self.scatter_back(self.out_hidden, residual, stream)

    def check(self, stream=None):
        code = up_read_status(self.status, stream)
        if code != 0:
            from . import up_status_string
            raise RuntimeError(f"device status {code}: {up_status_string(code, True)}")
