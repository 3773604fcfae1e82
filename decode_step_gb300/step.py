"""One batched decode step through the C ABI: append, attend, score and pick.

`DecodeStep` owns the workspaces and output buffers for a fixed batch shape
and issues tts_kv_append -> tts_decode_attn -> tts_codebook_head_select on one
stream.  The attention output [B][q_len][Hq][D] is read by the head as
h [B * q_len][Hq * D], so Hq * D must equal the head's hidden width.
"""
from __future__ import annotations

import math

import torch

from . import binding as bd


class DecodeStep:
    def __init__(self, cache: bd.KVCache, W: torch.Tensor, num_q_heads: int, B: int,
                 max_ctx_len: int, q_len: int = 1, causal: bool = False,
                 mode: int = bd.TTS_ARGMAX, temperature: float = 0.0, scale: float | None = None):
        dev = cache.k_pool.device
        self.cache, self.W = cache, W
        self.B, self.q_len, self.Hq = B, q_len, num_q_heads
        self.max_ctx_len, self.causal = max_ctx_len, causal
        self.mode, self.temperature = mode, temperature
        self.scale = 1.0 / math.sqrt(cache.head_dim) if scale is None else scale
        H = num_q_heads * cache.head_dim
        if W.shape[1] != H:
            raise ValueError(f"head width {W.shape[1]} != num_q_heads * head_dim = {H}")
        self.R, self.V = B * q_len, W.shape[0]
        attn_ws = bd.tts_decode_attn_workspace_size(B, q_len, num_q_heads, cache.num_kv_heads,
                                                    cache.head_dim, max_ctx_len)
        head_ws = bd.tts_head_workspace_size(self.R, self.V)
        if attn_ws == 0 or head_ws == 0:
            raise ValueError("unsupported decode-step shape")
        self.attn_ws = torch.zeros(attn_ws, dtype=torch.uint8, device=dev)
        self.head_ws = torch.zeros(head_ws, dtype=torch.uint8, device=dev)
        self.out = torch.empty((B, q_len, num_q_heads, cache.head_dim), dtype=cache.dtype, device=dev)
        self.ids = torch.empty(self.R, dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def __call__(self, block_table, ctx_before, ctx_lens, q, k_new, v_new, seed=None, step=None,
                 eos_allowed=None, logits_out=None, best=None, stream=None) -> torch.Tensor:
        """Runs the step; returns the device tensor of chosen ids [B * q_len]."""
        bd.tts_kv_append(self.cache, block_table, ctx_before, k_new, v_new, err=self.err, stream=stream)
        bd.tts_decode_attn(self.cache, block_table, ctx_lens, self.max_ctx_len, q, self.out,
                           self.attn_ws, self.scale, self.causal, err=self.err, stream=stream)
        h = self.out.view(self.R, self.Hq * self.cache.head_dim)
        bd.tts_codebook_head_select(h, self.W, self.ids, self.head_ws, mode=self.mode,
                                    temperature=self.temperature, seed=seed, step=step,
                                    eos_allowed=eos_allowed, best=best, logits_out=logits_out,
                                    stream=stream)
        return self.ids
