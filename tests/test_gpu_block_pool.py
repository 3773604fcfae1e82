"""The KV block pool on the step path: streams take their blocks from
tts_block_pool, run decode steps, two are aborted (barge-in), their blocks go
back to the pool and are poisoned with NaN on the device, and two new streams
receive exactly those blocks (the pool hands out the most recently freed ids
first) and run in the next batch ("Optimizing Streaming Text-to-Speech Models
for Sub-50 Millisecond Latency", section "Dynamic Token-Level Batching": a
static pool of 16-token blocks taken and returned per request; "TTS Serving,
in depth", section "Barge-in and cancellation").

The oracle never sees an id the library produced: the test keeps its own
model of the pool (a LIFO list of free ids), checks that the library hands
out the same ids, and gives the oracle the model's tables.  Every slot the
steps do not write holds NaN, so an attention that read a stale or foreign
slot would not stay finite.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import ATOL, as_f64, attn_errors, dev, host

pytestmark = pytest.mark.gpu

Hq, Hkv, D, BLK = 16, 8, 128, wl.BLOCK
NAN_BF16 = np.uint16(0x7FC0)


class PoolModel:
    """The pool's documented behaviour: a fresh pool hands out 0, 1, 2, ...;
    freed ids are handed out again last-freed-first."""

    def __init__(self, n):
        self.free = list(range(n - 1, -1, -1))   # top of the stack at the end

    def alloc(self, n):
        assert n <= len(self.free)
        out = [self.free.pop() for _ in range(n)]
        return out

    def release(self, ids):
        self.free.extend(ids)


def _rows(rng, n):
    return wl.f32_to_bf16(rng.standard_normal((1, n, Hkv, D), dtype=np.float32))


def _table(rows, width):
    t = np.full((len(rows), width), -1, dtype=np.int32)
    for b, r in enumerate(rows):
        t[b, :len(r)] = r
    return t


def test_barge_in_blocks_reused_without_stale_reads(orc, parity):
    from decode_step_gb300 import binding as bd
    rng = np.random.default_rng(4040)
    B = 10
    ctx = rng.integers(20, 300, size=B).astype(np.int32)    # lengths after this step's token
    need = [-(-int(L) // BLK) for L in ctx]
    nb = sum(need) + 6
    width = max(need) + 4
    pool, model = bd.BlockPool(nb), PoolModel(nb)
    blocks = []
    for n in need:
        got = pool.alloc(n)
        assert got == model.alloc(n), "pool order differs from last-freed-first"
        blocks.append(got)

    nan_pool = np.full((nb, Hkv, BLK, D), NAN_BF16, dtype=np.uint16)
    kp_h, vp_h = nan_pool.copy(), nan_pool.copy()                 # oracle pools
    kp_d, vp_d = dev(nan_pool), dev(nan_pool)                     # device pools
    cache = bd.KVCache(kp_d, vp_d)
    scale = 1.0 / math.sqrt(D)

    def prefill(b_rows, L_prompt):
        """Writes a prompt of L_prompt tokens through the append (q_len = L_prompt)."""
        t = _table([b_rows], width)
        k, v = _rows(rng, L_prompt), _rows(rng, L_prompt)
        z = np.zeros(1, dtype=np.int32)
        bd.tts_kv_append(cache, dev(t), dev(z), dev(k), dev(v))
        orc.kv_append(kp_h, vp_h, t, z, k, v, inplace=True)

    def step(rows, L, label):
        """One decode step over the batch: append the token at L - 1, attend."""
        n = len(rows)
        t = _table(rows, width)
        before = (L - 1).astype(np.int32)
        k, v = _rows(rng, n).reshape(n, 1, Hkv, D), _rows(rng, n).reshape(n, 1, Hkv, D)
        q = wl.f32_to_bf16(rng.standard_normal((n, 1, Hq, D), dtype=np.float32))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        td, Ld, qd = dev(t), dev(L.astype(np.int32)), dev(q)
        bd.tts_kv_append(cache, td, dev(before), dev(k), dev(v), err=err)
        ws = torch.zeros(bd.tts_decode_attn_workspace_size(n, 1, Hq, Hkv, D, int(L.max())), dtype=torch.uint8,
                         device="cuda")
        out = torch.empty_like(qd)
        bd.tts_decode_attn(cache, td, Ld, int(L.max()), qd, out, ws, scale, False, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        orc.kv_append(kp_h, vp_h, t, before, k, v, inplace=True)
        ref = orc.decode_attn(kp_h, vp_h, t, L, q, scale)
        got = as_f64(host(out), "bf16")
        assert np.isfinite(got).all(), f"{label}: non-finite output (a stale or foreign slot was read)"
        bad, mx_abs, mx_rel = attn_errors(got, ref)
        parity(f"block pool {label}", streams=n, max_abs=mx_abs, max_rel=mx_rel)
        assert bad == 0 and mx_abs <= ATOL, f"{label}: {bad} elements outside tolerance (max-abs {mx_abs})"

    for b in range(B):
        prefill(blocks[b], int(ctx[b]) - 1)
    step(blocks, ctx, "first step")
    # the cached bytes equal the oracle's pools wherever the steps wrote
    assert np.array_equal(host(kp_d), kp_h) and np.array_equal(host(vp_d), vp_h)

    # barge-in: streams 2 and 6 are aborted; their blocks go back to the pool
    # (stream 6 last, so its blocks come out first) and are poisoned
    aborted = [2, 6]
    freed = []
    for b in aborted:
        pool.free(blocks[b])
        model.release(blocks[b])
        freed += blocks[b]
    assert pool.num_free == len(model.free)
    idx = torch.tensor(freed, dtype=torch.long, device="cuda")
    kp_d[idx] = float("nan")
    vp_d[idx] = float("nan")
    kp_h[freed] = NAN_BF16
    vp_h[freed] = NAN_BF16

    # two new streams take blocks: most recently freed first
    new_ctx = np.array([BLK * len(blocks[6]) - 3, 17], dtype=np.int32)
    new_blocks = []
    for L in new_ctx:
        n = -(-int(L) // BLK)
        got = pool.alloc(n)
        assert got == model.alloc(n)
        new_blocks.append(got)
    assert set(new_blocks[0]) <= set(blocks[6]), "the first new stream should reuse the last freed blocks"
    for r, L in zip(new_blocks, new_ctx):
        prefill(r, int(L) - 1)

    # next step: the surviving streams (one token longer) and the new ones
    keep = [b for b in range(B) if b not in aborted]
    rows = [blocks[b] for b in keep] + new_blocks
    L2 = np.concatenate([ctx[keep] + 1, new_ctx]).astype(np.int32)
    for i, b in enumerate(keep):   # a survivor that crossed into a new block takes one from the pool
        while len(rows[i]) * BLK < L2[i]:
            extra = pool.alloc(1)
            assert extra == model.alloc(1)
            rows[i] = rows[i] + extra
    step(rows, L2, "after barge-in reuse")
    assert np.array_equal(host(kp_d), kp_h) and np.array_equal(host(vp_d), vp_h)
    pool.close()
