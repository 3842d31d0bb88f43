"""``MultiHeadAttention``: the sublayer as a module over the C ABI.

Mirrors the pages' MultiHeadedAttention(h, d_model) ("003-Transformer"
tutorial, section "Multi-head attention"): four Linear(d_model, d_model)
layers, forward(query, key, value, mask) -> [B, L_q, d_model], and the last
attention weights kept in ``self.attn`` when requested. PyTorch only holds the
device memory (weights, workspace, outputs) and the stream; every step of the
forward pass runs in libmha.so.
"""
from __future__ import annotations

import torch

from . import binding


class MultiHeadAttention:
    def __init__(self, h: int, d_model: int, *, dtype=torch.bfloat16, device="cuda", weights=None):
        if d_model % h != 0:
            raise ValueError(f"d_model ({d_model}) must be a multiple of h ({h})")
        self.h, self.d_model, self.dtype, self.device = h, d_model, dtype, torch.device(device)
        self.dt = binding.MHA_BF16 if dtype == torch.bfloat16 else binding.MHA_F32
        if weights is None:
            bound = (6.0 / (2 * d_model)) ** 0.5
            weights = {}
            for n in "qkvo":
                weights["w_" + n] = (torch.rand(d_model, d_model) * 2 - 1) * bound
                weights["b_" + n] = torch.zeros(d_model)
        self.weights = {k: torch.as_tensor(v).to(device=self.device, dtype=dtype).contiguous()
                        for k, v in weights.items()}
        self.attn = None
        self._ws = None

    def _workspace(self, B, Lq, Lk):
        need = binding.workspace_size(self.dt, B, Lq, Lk, self.d_model, self.h)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, query, key, value, *, causal=False, key_valid_lens=None, dense_mask=None,
                need_weights=False, out=None, stream=None):
        B, Lq, d = query.shape
        Lk = key.shape[1]
        w = self.weights
        vl = None if key_valid_lens is None else torch.as_tensor(
            key_valid_lens, dtype=torch.int32, device=self.device).contiguous()
        dm = None if dense_mask is None else torch.as_tensor(
            dense_mask, dtype=torch.uint8, device=self.device).contiguous()
        mask = binding.make_mask(causal, vl, dm)
        if out is None:
            out = torch.empty(B, Lq, d, dtype=self.dtype, device=self.device)
        p = torch.empty(B, self.h, Lq, Lk, dtype=torch.float32, device=self.device) if need_weights else None
        binding.mha_forward(query, key, value, w["w_q"], w["b_q"], w["w_k"], w["b_k"], w["w_v"], w["b_v"],
                            w["w_o"], w["b_o"], self.h, out=out, workspace=self._workspace(B, Lq, Lk),
                            mask=mask, p_attn=p, stream=stream)
        if need_weights:
            self.attn = p
        return out

    __call__ = forward
