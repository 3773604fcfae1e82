"""Seeded synthetic inputs for the batched codec-LM decode step.

This module draws random numbers and lays them out in the shapes the step
consumes. It computes none of the step's arithmetic (no attention, no logits,
no token selection); both the CPU oracle and the CUDA path are fed from here.

Workloads (shapes follow the pages' serving setting: a 12.5 Hz codec clock,
4 retained RVQ streams, tens of concurrent streams, 16-token KV blocks; see
"Optimizing Streaming Text-to-Speech Models for Sub-50 Millisecond Latency",
section "Dynamic Token-Level Batching", and "TontaubeV1", section 3):

  1 tiny       B=4,   Hq/Hkv=4/2,  D=64,  fp32, ctx U[16,64],     H=256  -> V=4097,  argmax
  2 semantic   B=16,  Hq/Hkv=16/8, D=128, bf16, ctx U[200,600],   H=2048 -> V=16385, argmax
  3 acoustic   B=64,  16/8, 128, bf16, ctx U[50,1500], permuted block table,  V=4097, argmax
  4 sampled    B=256, 16/8, 128, bf16, ctx log-U[32,4096],          V=16385, Gumbel T=0.7
  5 verify     B=64,  16/8, 128, bf16, q_len=5 causal, ctx U[256,2048], R=320 rows, V=4097,
               logits out, K=4 drafts, T=0.7

Every array is numpy. bf16 tensors are carried as their raw uint16 bit
patterns (numpy has no bfloat16); `bf16_to_f32` upcasts them exactly.

Pool slots that hold no context token (the tail of a stream's last block, the
slots the appended tokens will occupy, spare blocks) are filled with NaN, so a
kernel that reads a slot it should not read produces a non-finite output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

BLOCK = 16
NUMPY_SEED_BASE = 1000
PHILOX_SEED_MUL = 7919
BF16_NAN = np.uint16(0x7FC0)


@dataclass(frozen=True)
class Workload:
    id: int
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: str            # "f32" or "bf16"
    ctx_dist: str         # "uniform" or "loguniform"
    ctx_lo: int
    ctx_hi: int
    q_len: int
    causal: bool
    H: int                # head input width
    V: int                # vocab incl. the boundary token (index V-1)
    mode: str             # "argmax" or "gumbel"
    T: float              # sampling temperature (head Gumbel, verify target)
    logits_out: bool      # head also writes fp32 logits (verify path)
    K: int                # draft tokens per stream (0: no verify)
    permute_table: bool   # physical blocks drawn in random order

    @property
    def R(self) -> int:
        """Rows scored by the head: one per stream and query position."""
        return self.B * self.q_len

    @property
    def max_blocks(self) -> int:
        return -(-self.ctx_hi // BLOCK)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    1: Workload(1, "tiny-fp32", 4, 4, 2, 64, "f32", "uniform", 16, 64, 1, False,
                256, 4097, "argmax", 0.0, False, 0, False),
    2: Workload(2, "semantic-b16", 16, 16, 8, 128, "bf16", "uniform", 200, 600, 1, False,
                2048, 16385, "argmax", 0.0, False, 0, False),
    3: Workload(3, "acoustic-b64", 64, 16, 8, 128, "bf16", "uniform", 50, 1500, 1, False,
                2048, 4097, "argmax", 0.0, False, 0, True),
    4: Workload(4, "semantic-gumbel-b256", 256, 16, 8, 128, "bf16", "loguniform", 32, 4096, 1,
                False, 2048, 16385, "gumbel", 0.7, False, 0, False),
    5: Workload(5, "spec-verify-b64-k4", 64, 16, 8, 128, "bf16", "uniform", 256, 2048, 5, True,
                2048, 4097, "gumbel", 0.7, True, 4, False),
}


def custom(base: int | Workload, **changes) -> Workload:
    """A workload derived from a named one with some fields changed."""
    w = WORKLOADS[base] if isinstance(base, int) else base
    return replace(w, **changes)


# ---------------------------------------------------------------- bf16 bits

def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    out[np.isnan(x)] = BF16_NAN
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact upcast of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_to_f32(x) if dtype == "bf16" else np.asarray(x, dtype=np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def _nan(dtype: str):
    return BF16_NAN if dtype == "bf16" else np.float32(np.nan)


# ---------------------------------------------------------------- generator

def draw_ctx_lens(w: Workload, rng: np.random.Generator) -> np.ndarray:
    """Context length of each stream after this step's append."""
    if w.ctx_dist == "uniform":
        L = rng.integers(w.ctx_lo, w.ctx_hi + 1, size=w.B)
    elif w.ctx_dist == "loguniform":
        L = np.rint(np.exp(rng.uniform(math.log(w.ctx_lo), math.log(w.ctx_hi), size=w.B)))
    else:
        raise ValueError(w.ctx_dist)
    return np.clip(L, max(w.ctx_lo, w.q_len), w.ctx_hi).astype(np.int32)


def layout_blocks(ctx_lens: np.ndarray, max_blocks: int, spare: int, permute: bool,
                  rng: np.random.Generator):
    """Assign physical pool blocks to every stream's logical blocks.

    Returns (num_blocks, block_table[B][max_blocks] int32, unused entries -1).
    """
    nb = -(-ctx_lens.astype(np.int64) // BLOCK)
    num_blocks = int(nb.sum()) + spare
    ids = rng.permutation(num_blocks) if permute else np.arange(num_blocks)
    table = np.full((len(ctx_lens), max_blocks), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nb):
        table[b, :n] = ids[off:off + n]
        off += n
    return num_blocks, table


def fill_pool(num_blocks: int, Hkv: int, D: int, dtype: str, table: np.ndarray,
              n_valid: np.ndarray, rng: np.random.Generator) -> np.ndarray:
    """Pool [num_blocks][Hkv][16][D]; N(0,1) in each stream's first n_valid slots, NaN elsewhere."""
    vals = rng.standard_normal((num_blocks, Hkv, BLOCK, D), dtype=np.float32)
    valid = np.zeros((num_blocks, BLOCK), dtype=bool)
    for b, n in enumerate(n_valid):
        for i in range(-(-int(n) // BLOCK)):
            k = min(BLOCK, int(n) - i * BLOCK)
            valid[table[b, i], :k] = True
    pool = _store(vals, dtype)
    del vals
    pool[~np.broadcast_to(valid[:, None, :, None], pool.shape)] = _nan(dtype)
    return pool


def philox_keys(w: Workload, rows: int):
    """Per-row Philox key halves (seed, step) used by every random draw of the step."""
    seed = (PHILOX_SEED_MUL * (w.id + 1) + np.arange(rows)).astype(np.uint64)
    step = np.zeros(rows, dtype=np.uint64)
    return seed, step


def make_inputs(w: Workload | int, seed: int | None = None, ctx_lens=None,
                with_head: bool = True, with_verify: bool | None = None) -> dict:
    """All inputs of one decode step of workload `w`, drawn from one seeded stream.

    Keys: ctx_lens, ctx_before, num_blocks, block_table, k_pool, v_pool, q,
    k_new, v_new, scale; with_head adds h, W, seed, step; with_verify adds
    target_logits, draft_probs, draft_tokens, vseed, vstep.
    """
    if isinstance(w, int):
        w = WORKLOADS[w]
    rng = np.random.default_rng(NUMPY_SEED_BASE + w.id if seed is None else seed)
    L = draw_ctx_lens(w, rng) if ctx_lens is None else np.asarray(ctx_lens, dtype=np.int32)
    assert L.shape == (w.B,) and int(L.min()) >= w.q_len and int(L.max()) <= w.ctx_hi
    ctx_before = (L - w.q_len).astype(np.int32)
    num_blocks, table = layout_blocks(L, w.max_blocks, spare=max(2, w.B // 4),
                                      permute=w.permute_table, rng=rng)
    out = dict(workload=w, ctx_lens=L, ctx_before=ctx_before, num_blocks=num_blocks,
               block_table=table, scale=1.0 / math.sqrt(w.D))
    qs = (w.B, w.q_len, w.Hq, w.D)
    ks = (w.B, w.q_len, w.Hkv, w.D)
    out["q"] = _store(rng.standard_normal(qs, dtype=np.float32), w.dtype)
    out["k_new"] = _store(rng.standard_normal(ks, dtype=np.float32), w.dtype)
    out["v_new"] = _store(rng.standard_normal(ks, dtype=np.float32), w.dtype)
    out["k_pool"] = fill_pool(num_blocks, w.Hkv, w.D, w.dtype, table, ctx_before, rng)
    out["v_pool"] = fill_pool(num_blocks, w.Hkv, w.D, w.dtype, table, ctx_before, rng)
    if with_head:
        out["h"] = _store(rng.standard_normal((w.R, w.H), dtype=np.float32), w.dtype)
        out["W"] = _store(0.02 * rng.standard_normal((w.V, w.H), dtype=np.float32), w.dtype)
        out["seed"], out["step"] = philox_keys(w, w.R)
    if with_verify is None:
        with_verify = w.K > 0
    if with_verify:
        K = w.K
        out["target_logits"] = rng.standard_normal((w.B, K + 1, w.V), dtype=np.float32)
        out["draft_probs"], out["draft_tokens"] = draft_model_outputs(w.B, K, w.V, rng)
        out["vseed"], out["vstep"] = philox_keys(w, w.B)
    return out


def draft_model_outputs(B: int, K: int, V: int, rng: np.random.Generator):
    """Stand-in for a draft model: probabilities from N(0,1) logits (T=1) and
    K proposed tokens per stream drawn from them (inverse CDF)."""
    x = rng.standard_normal((B, K, V)).astype(np.float64)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    probs = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    cdf = np.cumsum(probs.astype(np.float64), axis=-1)
    u = rng.random((B, K, 1)) * cdf[..., -1:]
    tokens = np.minimum((cdf < u).sum(axis=-1), V - 1).astype(np.int32)
    return probs, tokens


# Two-layer audio head ("TontaubeV1", section 3): the transformer state is
# expanded to width 4,096 through Mish, then projected to the stage's
# vocabulary, whose last ids are the stage's structural tokens.
AUDIO_HEAD_SHAPES = {
    # name: (R, H, F, V, n_tail)
    "acoustic-b64": (64, 2048, 4096, 4097, 1),   # an acoustic stage: 4,096 codes + the boundary
    "semantic-cb0-b16": (16, 2048, 4096, 16386, 2),  # CB0: 16,384 codes + row terminator + <|audio_split|>
}


def audio_head_inputs(R: int, H: int, F: int, V: int, n_tail: int, seed: int = 4242) -> dict:
    """Seeded inputs of the two-layer audio head: state h ~ N(0, 1); weights
    and biases of both layers uniform in +-1/sqrt(fan_in), the usual
    initialisation of a fresh linear layer (the pages' heads are newly
    initialised; no trained weights exist here); per-row mask bits of the
    structural tail drawn uniformly; Philox keys per row."""
    rng = np.random.default_rng(seed)
    a1, a2 = 1.0 / math.sqrt(H), 1.0 / math.sqrt(F)
    out = dict(
        h=f32_to_bf16(rng.standard_normal((R, H), dtype=np.float32)),
        W1=f32_to_bf16(rng.uniform(-a1, a1, (F, H)).astype(np.float32)),
        b1=rng.uniform(-a1, a1, F).astype(np.float32),
        W2=f32_to_bf16(rng.uniform(-a2, a2, (V, F)).astype(np.float32)),
        b2=rng.uniform(-a2, a2, V).astype(np.float32),
        tail_allowed=rng.integers(0, 1 << n_tail, R).astype(np.uint32) if n_tail else np.zeros(R, np.uint32),
        seed=(PHILOX_SEED_MUL * 97 + np.arange(R)).astype(np.uint64),
        step=np.zeros(R, dtype=np.uint64),
    )
    return out


# Code predictor ("How We Made a TTS Model Respond in Sub-50 ms": a fixed loop
# of autoregressive steps per frame, one per remaining codebook, over a short
# bounded context).  The pages give no architecture; the loop here is one
# projection, attention and codebook head per step.
CODE_PREDICTOR = dict(R=64, H=1024, Hq=8, Hkv=4, D=128, V=2048, n_steps=15)


def code_predictor_inputs(R: int, H: int, Hq: int, Hkv: int, D: int, V: int, n_steps: int,
                          seed: int = 5150) -> dict:
    """Seeded inputs of the predictor's frame loop: the talker's states
    x0 ~ N(0, 1); projection and per-codebook head weights uniform in
    +-1/sqrt(H) (a fresh linear layer's initialisation); codebook embeddings
    ~ N(0, 1); all bf16.  Philox keys per stream (step = the frame index)."""
    rng = np.random.default_rng(seed)
    a = 1.0 / math.sqrt(H)
    F = (Hq + 2 * Hkv) * D
    return dict(
        x0=f32_to_bf16(rng.standard_normal((R, H), dtype=np.float32)),
        Wqkv=f32_to_bf16(rng.uniform(-a, a, (F, H)).astype(np.float32)),
        W=f32_to_bf16(rng.uniform(-a, a, (n_steps, V, Hq * D)).astype(np.float32)),
        E=f32_to_bf16(rng.standard_normal((n_steps, V, H), dtype=np.float32)),
        seed=(PHILOX_SEED_MUL * 131 + np.arange(R)).astype(np.uint64),
        step=np.full(R, 3, dtype=np.uint64),
    )
