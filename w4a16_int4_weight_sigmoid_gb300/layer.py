"""Device-resident W4A16 MoE layer: prepacked weights + workspace + one call.

Memory management and marshalling only (torch allocates, the library
computes): weights are uploaded once and repacked on the device by
chord_w4a16_prepack; forward() is one chord_moe_layer call.
"""
from __future__ import annotations

import numpy as np
import torch

from . import chord


def to_device(a, device="cuda"):
    """numpy array -> torch tensor on device (uint16 arrays become bfloat16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def prepack(q, s, gate_up: bool, stream=None):
    """Device uint8 [E,N,K/2] + bfloat16 [E,N,K/32] -> packed blob (uint8 tensor)."""
    E, N, K2 = q.shape
    nbytes = chord.chord_w4a16_prepack_bytes(E, N, 2 * K2)
    packed = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    chord.chord_w4a16_prepack(q, s, gate_up, packed, stream=stream)
    return packed


class W4A16MoELayer:
    """One expert shard of a MoE layer (local experts [expert_begin, +E_local))."""

    def __init__(self, w13_q, w13_s, w2_q, w2_s, E_total: int, expert_begin: int, topk: int,
                 device="cuda"):
        w13_q, w13_s = to_device(w13_q, device), to_device(w13_s, device)
        w2_q, w2_s = to_device(w2_q, device), to_device(w2_s, device)
        self.E_local, twoI, H2 = w13_q.shape
        self.H, self.I = 2 * H2, twoI // 2
        self.E_total, self.expert_begin, self.topk = E_total, expert_begin, topk
        self.w13 = prepack(w13_q, w13_s, True)
        self.w2 = prepack(w2_q, w2_s, False)
        torch.cuda.synchronize()
        self._ws = None
        self._ws_M = -1
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)

    def workspace(self, M: int):
        if M > self._ws_M:
            n = chord.chord_moe_layer_workspace_bytes(M, self.H, self.I, self.E_local, self.topk)
            self._ws = torch.empty(max(n, 1), dtype=torch.uint8, device=self.w13.device)
            self._ws_M = M
        return self._ws

    def forward(self, x, logits, bias, out=None, topk_weights_out=None, topk_ids_out=None,
                tuning=None, stream=None):
        M = x.shape[0]
        if out is None:
            out = torch.empty((M, self.H), dtype=torch.bfloat16, device=x.device)
        chord.chord_moe_layer(x, logits, bias, self.w13, self.w2, self.H, self.I, self.E_total,
                              self.expert_begin, self.E_local, self.topk, out, self.workspace(M),
                              topk_weights_out, topk_ids_out, tuning=tuning,
                              dev_status=self.dev_status, stream=stream)
        return out
