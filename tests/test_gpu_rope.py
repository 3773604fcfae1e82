"""Append with the rotary embedding fused in (tts_kv_append_rope), against the oracle.

The oracle rotates in double and rounds once; the kernel takes cos and sin
from double precision, rounds them to fp32 and rotates in fp32, so its rotated
value is within a few fp32 ulps of the oracle's.  A stored bf16 or e4m3 value
may therefore differ from the oracle's rounding only where the oracle's value
sits that close to the midpoint between two representable neighbours; every
other element, every value row and every untouched byte must match exactly.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import attn_errors, dev, host
from oracle_pins import fp8_tile_views
from test_gpu_fp8 import fp8_cache_for

pytestmark = pytest.mark.gpu

# Bound on |kernel - oracle| for a rotated value, relative to |x_i| + |x_{i+64}|
# (cos/sin rounded to fp32, two products and an fma: a few 2^-24).
ROT_TOL = 2.0 ** -20
ERR_INVALID, ERR_UNSUPPORTED = -1, -2   # status codes of the C interface


@pytest.fixture(scope="module")
def bd():
    from decode_step_gb300 import binding
    return binding


CASES = [
    # (base workload, changes)
    (3, dict(B=8, ctx_lo=20, ctx_hi=300)),
    (3, dict(B=5, ctx_lo=1, ctx_hi=40, lens=[1, 2, 17, 33, 40])),  # position 0: the identity
    (5, dict(B=4, ctx_lo=6, ctx_hi=200)),            # q_len 5
    (3, dict(B=3, Hq=16, Hkv=4, ctx_lo=1500, ctx_hi=2040)),
    (3, dict(B=3, Hq=8, Hkv=8, ctx_lo=30, ctx_hi=120)),
]
IDS = [f"c{i}" for i in range(len(CASES))]


def _inputs(base, changes, seed):
    changes = dict(changes)
    lens = changes.pop("lens", None)
    w = wl.custom(base, **changes, permute_table=True)
    return wl.make_inputs(w, seed=seed, with_head=False, with_verify=False,
                          ctx_lens=None if lens is None else np.array(lens, np.int32))


def _positions(inp):
    w = inp["workload"]
    return inp["ctx_before"][:, None].astype(np.int64) + np.arange(w.q_len)[None, :]


def _pair_mag(x_bits):
    """|x_i| + |x_{i+64}| for every element of rows x [..., 128] (bf16 bits)."""
    x = np.abs(wl.bf16_to_f32(x_bits).astype(np.float64))
    h = x.shape[-1] // 2
    m = x[..., :h] + x[..., h:]
    return np.concatenate([m, m], axis=-1)


def check_bf16_rounding(got_bits, y, mag, what):
    """got_bits equals round-to-nearest-bf16(y) except where y lies within
    ROT_TOL * mag of the midpoint between the two bf16 neighbours got differs by."""
    exp = wl.f32_to_bf16(y.astype(np.float32))
    bad = np.nonzero(got_bits != exp)
    n = len(bad[0])
    if n:
        g = wl.bf16_to_f32(got_bits[bad]).astype(np.float64)
        e = wl.bf16_to_f32(exp[bad]).astype(np.float64)
        yy = y[bad].astype(np.float64)
        ulp = np.abs(e) * 2.0 ** -7 + 1e-45
        near = (np.abs(g - e) <= ulp) & (np.abs(yy - 0.5 * (g + e)) <= ROT_TOL * mag[bad] + 1e-30)
        assert near.all(), f"{what}: {int((~near).sum())} elements off by more than a rounding tie"
    print(f"[rope {what}] {n} of {got_bits.size} roundings taken the other way at a tie")
    return n


def e4m3_values():
    """Decoded value of every finite e4m3 code (NaN for 0x7F / 0xFF)."""
    c = np.arange(256, dtype=np.uint8)
    s = np.where(c >> 7, -1.0, 1.0)
    e, m = (c >> 3) & 15, (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8) * 2.0 ** (e.astype(np.float64) - 7))
    v = s * mag
    v[(e == 15) & (m == 7)] = np.nan
    return v


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_rope_append_bf16(orc, bd, case):
    inp = _inputs(*case, seed=900 + CASES.index(case))
    w = inp["workload"]
    pos = _positions(inp)
    q_rot = orc.rope(inp["q"], pos)
    k_rot = orc.rope(inp["k_new"], pos)
    ref_k, ref_v = orc.kv_append(inp["k_pool"], inp["v_pool"], inp["block_table"], inp["ctx_before"],
                                 wl.f32_to_bf16(k_rot), inp["v_new"])
    kp, vp = dev(inp["k_pool"]), dev(inp["v_pool"])
    cache = bd.KVCache(kp, vp)
    q = dev(inp["q"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_kv_append_rope(cache, dev(inp["block_table"]), dev(inp["ctx_before"]), q, dev(inp["k_new"]),
                          dev(inp["v_new"]), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(host(vp), ref_v)
    check_bf16_rounding(host(q), q_rot, _pair_mag(inp["q"]), "q")
    # key rows: the slots written this step, compared with rounding ties allowed;
    # every other slot exactly
    got_k = host(kp)
    t = pos.reshape(-1)
    b = np.repeat(np.arange(w.B), w.q_len)
    blocks, slots = inp["block_table"][b, t // wl.BLOCK], t % wl.BLOCK
    written = np.zeros(got_k.shape[:1] + got_k.shape[2:3], bool)
    written[blocks, slots] = True
    other = ~written[:, None, :, None] & np.ones(got_k.shape, bool)
    assert np.array_equal(got_k[other], ref_k[other])
    rows = got_k[blocks, :, slots, :].reshape(w.B, w.q_len, w.Hkv, w.D)
    check_bf16_rounding(rows, k_rot, _pair_mag(inp["k_new"]), "k")
    if min(pos.reshape(-1)) == 0:  # position 0 rotates nothing
        z = pos == 0
        assert np.array_equal(rows[z], inp["k_new"][z])


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_rope_append_fp8(orc, bd, case):
    inp = _inputs(*case, seed=950 + CASES.index(case))
    w = inp["workload"]
    pos = _positions(inp)
    q_rot = orc.rope(inp["q"], pos)
    k_rot = orc.rope(inp["k_new"], pos)
    tiles = fp8_cache_for(orc, inp)
    ref = orc.kv_append_fp8(tiles, inp["block_table"], inp["ctx_before"], k_rot,
                            wl.bf16_to_f32(inp["v_new"]))
    cache = bd.KVCache(dev(tiles))
    q = dev(inp["q"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_kv_append_rope(cache, dev(inp["block_table"]), dev(inp["ctx_before"]), q, dev(inp["k_new"]),
                          dev(inp["v_new"]), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_bf16_rounding(host(q), q_rot, _pair_mag(inp["q"]), "q")
    got = host(cache.k_pool)
    gk, gv, gks, gvs = fp8_tile_views(got)
    rk, rv, rks, rvs = fp8_tile_views(ref)
    # value codes, value scales and the untouched slots' bytes: exact
    assert np.array_equal(gv, rv)
    assert np.array_equal(gvs.view(np.uint32), rvs.view(np.uint32))
    t = pos.reshape(-1)
    b = np.repeat(np.arange(w.B), w.q_len)
    blocks, slots = inp["block_table"][b, t // wl.BLOCK], t % wl.BLOCK
    written = np.zeros((got.shape[0], wl.BLOCK), bool)
    written[blocks, slots] = True
    keep = ~written[:, None, :] & np.ones(gks.shape, bool)
    assert np.array_equal(gk[keep], rk[keep])
    assert np.array_equal(gks.view(np.uint32)[keep], rks.view(np.uint32)[keep])
    # written key rows: scale within the rotation's error, codes equal to the
    # oracle's except at a rounding tie of x / scale
    gs = gks[blocks, :, slots].reshape(w.B, w.q_len, w.Hkv).astype(np.float64)
    rs = rks[blocks, :, slots].reshape(w.B, w.q_len, w.Hkv).astype(np.float64)
    mag = _pair_mag(inp["k_new"])
    assert np.all(np.abs(gs - rs) <= 4 * ROT_TOL * mag.max(axis=-1) / 448 + 1e-30)
    gc = gk[blocks, :, slots].reshape(w.B, w.q_len, w.Hkv, w.D)
    rc = rk[blocks, :, slots].reshape(w.B, w.q_len, w.Hkv, w.D)
    bad = np.nonzero(gc != rc)
    n = len(bad[0])
    if n:
        val = e4m3_values()
        g, e = val[gc[bad]], val[rc[bad]]
        x = k_rot[bad].astype(np.float64) / rs[bad[:3]]
        # adjacent codes and x / scale within the rotation's error of their midpoint
        step = np.abs(np.abs(g) - np.abs(e))
        assert np.all(np.sign(g) * np.sign(e) >= 0) and np.all(step <= np.maximum(np.abs(e), 2.0 ** -6) / 8 + 1e-12)
        tol = 2 * ROT_TOL * mag[bad] / rs[bad[:3]] + 4 * ROT_TOL * np.abs(x)
        assert np.all(np.abs(x - 0.5 * (g + e)) <= tol)
    print(f"[rope fp8 k] {n} of {gc.size} codes taken the other way at a tie")


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_rope_then_attention(orc, bd, fp8):
    """Rotated append followed by attention on the rotated queries matches the
    oracle's rotation, append and attention."""
    inp = _inputs(5, dict(B=6, ctx_lo=40, ctx_hi=700), seed=990 + fp8)
    w = inp["workload"]
    pos = _positions(inp)
    q_rot = wl.f32_to_bf16(orc.rope(inp["q"], pos))
    k_rot = orc.rope(inp["k_new"], pos)
    scale = 1.0 / math.sqrt(w.D)
    if fp8:
        tiles = fp8_cache_for(orc, inp)
        ref_tiles = orc.kv_append_fp8(tiles, inp["block_table"], inp["ctx_before"], k_rot,
                                      wl.bf16_to_f32(inp["v_new"]))
        ref = orc.decode_attn_fp8(ref_tiles, inp["block_table"], inp["ctx_lens"], q_rot, scale, w.causal)
        cache = bd.KVCache(dev(tiles))
    else:
        rk, rv = orc.kv_append(inp["k_pool"], inp["v_pool"], inp["block_table"], inp["ctx_before"],
                               wl.f32_to_bf16(k_rot), inp["v_new"])
        ref = orc.decode_attn(rk, rv, inp["block_table"], inp["ctx_lens"], q_rot, scale, w.causal)
        cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
    table = dev(inp["block_table"])
    q = dev(inp["q"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_kv_append_rope(cache, table, dev(inp["ctx_before"]), q, dev(inp["k_new"]), dev(inp["v_new"]), err=err)
    out = torch.empty((w.B, w.q_len, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(bd.tts_decode_attn_workspace_size(w.B, w.q_len, w.Hq, w.Hkv, w.D, w.ctx_hi),
                     dtype=torch.uint8, device="cuda")
    bd.tts_decode_attn(cache, table, dev(inp["ctx_lens"]), w.ctx_hi, q, out, ws, scale, w.causal, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = wl.bf16_to_f32(host(out)).astype(np.float64)
    bad, emax, rel = attn_errors(got, ref)
    print(f"[rope attn fp8={fp8}] max abs {emax:.3g} max rel {rel:.3g} failing {bad}")
    assert bad == 0


def test_rope_append_errors(bd):
    """Argument checks: an fp32 cache is unsupported; a base <= 1, NaN or infinite is invalid."""
    inp = _inputs(1, dict(B=2, ctx_lo=3, ctx_hi=20), seed=5)
    w = inp["workload"]
    cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
    q = torch.zeros((w.B, w.q_len, w.Hq, w.D), dtype=torch.float32, device="cuda")
    with pytest.raises(bd.TTSError) as e:
        bd.tts_kv_append_rope(cache, dev(inp["block_table"]), dev(inp["ctx_before"]), q, dev(inp["k_new"]),
                              dev(inp["v_new"]))
    assert e.value.code == ERR_UNSUPPORTED
    inp = _inputs(3, dict(B=2, ctx_lo=3, ctx_hi=20), seed=6)
    w = inp["workload"]
    cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
    args = (cache, dev(inp["block_table"]), dev(inp["ctx_before"]), dev(inp["q"]), dev(inp["k_new"]),
            dev(inp["v_new"]))
    for base in (1.0, 0.5, float("nan"), float("inf")):
        with pytest.raises(bd.TTSError) as e:
            bd.tts_kv_append_rope(*args, rope_base=base)
        assert e.value.code == ERR_INVALID


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_rope_decode_step_ids(orc, bd, fp8):
    """The fused step with the rotation (tts_decode_step, rope_base != 0) and its
    captured form: ids as the oracle head picks them on the oracle's attention
    over the oracle-rotated queries and keys."""
    from decode_step_gb300.step import DecodeStep, GraphedStep
    from gpu_util import compare_ids
    w = wl.custom(3, B=16, ctx_lo=30, ctx_hi=400, permute_table=True)
    inp = wl.make_inputs(w, seed=1234 + fp8, with_verify=False)
    pos = _positions(inp)
    q_rot = wl.f32_to_bf16(orc.rope(inp["q"], pos))
    k_rot = orc.rope(inp["k_new"], pos)
    if fp8:
        tiles = fp8_cache_for(orc, inp)
        ref_tiles = orc.kv_append_fp8(tiles, inp["block_table"], inp["ctx_before"], k_rot,
                                      wl.bf16_to_f32(inp["v_new"]))
        attn = orc.decode_attn_fp8(ref_tiles, inp["block_table"], inp["ctx_lens"], q_rot, inp["scale"])
        cache = bd.KVCache(dev(tiles))
    else:
        rk, rv = orc.kv_append(inp["k_pool"], inp["v_pool"], inp["block_table"], inp["ctx_before"],
                               wl.f32_to_bf16(k_rot), inp["v_new"])
        attn = orc.decode_attn(rk, rv, inp["block_table"], inp["ctx_lens"], q_rot, inp["scale"])
        cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
    h = wl.f32_to_bf16(attn.reshape(w.R, w.Hq * w.D).astype(np.float32))
    ref = orc.head_select(h, inp["W"], "argmax")
    step = DecodeStep(cache, dev(inp["W"]), w.Hq, w.B, w.ctx_hi, rope_base=10000.0)
    table, cb, cl = dev(inp["block_table"]), dev(inp["ctx_before"]), dev(inp["ctx_lens"])
    q, kn, vn = dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"])
    ids = step(table, cb, cl, q, kn, vn).clone()
    torch.cuda.synchronize()
    check_bf16_rounding(host(q), orc.rope(inp["q"], pos), _pair_mag(inp["q"]), "step q")
    hard, ties = compare_ids(host(ids), ref)
    print(f"[rope step fp8={fp8}] near-ties {ties}, hard mismatches {len(hard)}")
    assert not hard
    # captured: every launch copies the unrotated q from pinned memory and rotates it again
    g = GraphedStep(step, {"block_table": table, "ctx_before": cb, "ctx_lens": cl, "q": dev(inp["q"]),
                           "k_new": kn, "v_new": vn})
    for _ in range(2):
        assert torch.equal(g().clone(), ids.cpu())
    assert int(step.err.item()) == 0
