"""FP8 E4M3 KV cache on the GPU against the oracle.

The cache a step starts from is the workload's context (the bf16 rows it
caches before this step) quantised by the oracle; slots holding no token keep
NaN codes and NaN scales, so a kernel that reads one produces a non-finite
output.  The append must match the oracle byte for byte; attention within the
attention tolerance; the fused step's ids match the oracle head on the
oracle's attention output except at near-ties.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import attn_errors, compare_ids, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bd():
    from decode_step_gb300 import binding
    return binding


def fp8_cache_for(orc, inp):
    """The context cached before this step, quantised into FP8 tiles by the
    oracle; every other code is NaN (0x7F) and every other scale NaN."""
    w = inp["workload"]
    nb, table = inp["num_blocks"], inp["block_table"]
    tiles = np.full((nb, w.Hkv, 4224), 0x7F, np.uint8)
    tiles[:, :, 4096:] = np.full(32, np.nan, np.float32).view(np.uint8)
    for b in range(w.B):
        n = int(inp["ctx_before"][b])
        if n == 0:
            continue
        t = np.arange(n)
        blocks, slots = table[b, t // wl.BLOCK], t % wl.BLOCK
        krows = np.ascontiguousarray(inp["k_pool"][blocks, :, slots, :])[None]
        vrows = np.ascontiguousarray(inp["v_pool"][blocks, :, slots, :])[None]
        tiles = orc.kv_append_fp8(tiles, table[b:b + 1], np.zeros(1, np.int32), krows, vrows)
    return tiles


def upload_cache(bd, tiles):
    return bd.KVCache(dev(tiles))


CASES = [
    # (base workload, changes)
    (3, dict(B=8, ctx_lo=20, ctx_hi=300)),
    (3, dict(B=5, ctx_lo=1, ctx_hi=40)),
    (5, dict(B=4, ctx_lo=6, ctx_hi=200)),
    (3, dict(B=3, Hq=16, Hkv=4, ctx_lo=30, ctx_hi=120)),   # group 4
    (3, dict(B=3, Hq=8, Hkv=8, ctx_lo=30, ctx_hi=120)),    # one query row per KV head
]


def _inputs(base, changes, seed):
    w = wl.custom(base, **changes, permute_table=True)
    return wl.make_inputs(w, seed=seed, with_head=False, with_verify=False)


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_fp8_append_matches_oracle_bytes(orc, bd, case):
    inp = _inputs(*case, seed=500 + CASES.index(case))
    w = inp["workload"]
    k_new, v_new = inp["k_new"].copy(), inp["v_new"].copy()
    k_new[0, 0, 0] = 0                                   # an all-zero row: scale 0, codes 0
    v_new[-1, -1, -1, :4] = wl.f32_to_bf16(np.array([3e38, -3e38, 1e-30, 0], np.float32))
    tiles = fp8_cache_for(orc, inp)
    ref = orc.kv_append_fp8(tiles, inp["block_table"], inp["ctx_before"], k_new, v_new)
    cache = upload_cache(bd, tiles)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_kv_append(cache, dev(inp["block_table"]), dev(inp["ctx_before"]), dev(k_new), dev(v_new), err=err)
    torch.cuda.synchronize()
    assert np.array_equal(host(cache.k_pool), ref)
    assert int(err.item()) == 0


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_fp8_attention_matches_oracle(orc, bd, case):
    inp = _inputs(*case, seed=600 + CASES.index(case))
    w = inp["workload"]
    tiles = orc.kv_append_fp8(fp8_cache_for(orc, inp), inp["block_table"], inp["ctx_before"], inp["k_new"],
                              inp["v_new"])
    cache = upload_cache(bd, tiles)
    out = torch.empty((w.B, w.q_len, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(bd.tts_decode_attn_workspace_size(w.B, w.q_len, w.Hq, w.Hkv, w.D, w.ctx_hi),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(w.D)
    for _ in range(2):  # twice: the workspace is left ready for the next call
        bd.tts_decode_attn(cache, dev(inp["block_table"]), dev(inp["ctx_lens"]), w.ctx_hi, dev(inp["q"]), out, ws,
                           scale, w.causal, err=err)
        torch.cuda.synchronize()
        ref = orc.decode_attn_fp8(tiles, inp["block_table"], inp["ctx_lens"], inp["q"], scale, w.causal)
        got = wl.bf16_to_f32(host(out)).astype(np.float64)
        assert np.isfinite(got).all()
        bad, emax, rel = attn_errors(got, ref)
        print(f"[fp8 attn {w.name} B={w.B}] max abs {emax:.3g} max rel {rel:.3g} failing {bad}")
        assert bad == 0
    assert int(err.item()) == 0


MAGNITUDES = [
    # (base workload, changes, value factor: a power of two, or "mixed" per row)
    (3, dict(B=6, ctx_lo=20, ctx_hi=300), 2.0 ** -12),
    (3, dict(B=6, ctx_lo=20, ctx_hi=300), 2.0 ** 14),
    (3, dict(B=6, ctx_lo=20, ctx_hi=300), "mixed"),
    (5, dict(B=4, ctx_lo=6, ctx_hi=200), "mixed"),
]


@pytest.mark.parametrize("case", MAGNITUDES, ids=[f"m{i}" for i in range(len(MAGNITUDES))])
def test_fp8_attention_value_magnitudes(orc, bd, case):
    """Values far from unit size (value scales from about 2^-20 up to 2^7.5,
    just below the interface's limit of 256), all alike or a different power
    of two per row (2^-6 .. 2^6): each output element is within 1% of itself
    plus 1% of the same attention over |V| (the scale of the sum it comes
    from), so the test does not depend on the values' size."""
    base, changes, factor = case
    inp = _inputs(base, changes, seed=650 + MAGNITUDES.index(case))
    w = inp["workload"]
    rng = np.random.default_rng(651 + MAGNITUDES.index(case))
    for key in ("v_pool", "v_new"):                 # powers of two keep bf16 values exact
        v = wl.bf16_to_f32(inp[key])
        f = 2.0 ** rng.integers(-6, 7, size=v.shape[:-1] + (1,)) if factor == "mixed" else factor
        inp[key] = wl.f32_to_bf16((v * f).astype(np.float32))
    vmax = np.nanmax(np.abs(wl.bf16_to_f32(inp["v_pool"])))
    assert vmax / 448 < 256                           # inside the interface's range
    tiles = orc.kv_append_fp8(fp8_cache_for(orc, inp), inp["block_table"], inp["ctx_before"], inp["k_new"],
                              inp["v_new"])
    cache = upload_cache(bd, tiles)
    out = torch.empty((w.B, w.q_len, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(bd.tts_decode_attn_workspace_size(w.B, w.q_len, w.Hq, w.Hkv, w.D, w.ctx_hi),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(w.D)
    bd.tts_decode_attn(cache, dev(inp["block_table"]), dev(inp["ctx_lens"]), w.ctx_hi, dev(inp["q"]), out, ws,
                       scale, w.causal, err=err)
    torch.cuda.synchronize()
    ref = orc.decode_attn_fp8(tiles, inp["block_table"], inp["ctx_lens"], inp["q"], scale, w.causal)
    absv = tiles.copy()
    absv[:, :, 2048:4096] &= 0x7F                    # |code|; the NaN code 0x7F stays NaN
    mag = orc.decode_attn_fp8(absv, inp["block_table"], inp["ctx_lens"], inp["q"], scale, w.causal)
    got = wl.bf16_to_f32(host(out)).astype(np.float64)
    assert np.isfinite(got).all()
    e = np.abs(got - ref)
    ok = e <= 1e-2 * (np.abs(ref) + mag)
    print(f"[fp8 attn magnitudes {factor}] max error / |V| attention {float((e / mag).max()):.3g}")
    assert ok.all(), f"{int((~ok).sum())} elements off"
    assert int(err.item()) == 0


def test_fp8_decode_step_ids(orc, bd):
    """The fused step on an FP8 cache: GPU append, attention and head; ids as
    the oracle head picks them on the oracle's attention output (bf16)."""
    from decode_step_gb300.step import DecodeStep, GraphedStep
    w = wl.custom(3, B=16, ctx_lo=30, ctx_hi=400, permute_table=True)
    inp = wl.make_inputs(w, seed=777, with_verify=False)
    tiles = fp8_cache_for(orc, inp)
    cache = upload_cache(bd, tiles)
    step = DecodeStep(cache, dev(inp["W"]), w.Hq, w.B, w.ctx_hi)
    table, cb, cl = dev(inp["block_table"]), dev(inp["ctx_before"]), dev(inp["ctx_lens"])
    q, kn, vn = dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"])
    ids = step(table, cb, cl, q, kn, vn).clone()
    torch.cuda.synchronize()
    ref_tiles = orc.kv_append_fp8(tiles, inp["block_table"], inp["ctx_before"], inp["k_new"], inp["v_new"])
    assert np.array_equal(host(cache.k_pool), ref_tiles)
    attn = orc.decode_attn_fp8(ref_tiles, inp["block_table"], inp["ctx_lens"], inp["q"], inp["scale"])
    h = wl.f32_to_bf16(attn.reshape(w.R, w.Hq * w.D).astype(np.float32))
    ref = orc.head_select(h, inp["W"], "argmax")
    hard, ties = compare_ids(host(ids), ref)
    print(f"[fp8 step] near-ties {ties}, hard mismatches {len(hard)}")
    assert not hard
    # the captured step gives the same ids
    g = GraphedStep(step, {"block_table": table, "ctx_before": cb, "ctx_lens": cl, "q": q, "k_new": kn, "v_new": vn})
    assert torch.equal(g().clone(), ids.cpu())
    assert int(step.err.item()) == 0
