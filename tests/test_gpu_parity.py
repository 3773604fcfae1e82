"""CUDA path against the CPU oracle, through the C ABI (needs a GB300).

Every workload at full size, plus small ragged shapes and edge cases.  The
bar: KV append bit-exact; attention within max(2e-2, 1e-2 |o|) per element
(fp32: 1e-4); token ids and accepted counts bit-exact except at near-ties
(oracle's top two keys, or acceptance ratio and uniform, closer than 1e-3),
which are counted and reported.
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import (ATOL, NEAR_TIE, RTOL, Uploaded, as_f64, attn_errors, compare_ids, dev, host,
                      rel_where_binding)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from decode_step_gb300 import binding as bd
    from decode_step_gb300.step import DecodeStep, GraphedStep


# ------------------------------------------------------------------ helpers

def gpu_append(u: Uploaded, err=None):
    cache = bd.KVCache(u.k_pool, u.v_pool)
    bd.tts_kv_append(cache, u.table, u.ctx_before, u.k_new, u.v_new, err=err)
    return cache


def gpu_attn(u: Uploaded, cache, max_ctx=None, err=None, q=None):
    w = u.w
    max_ctx = w.ctx_hi if max_ctx is None else max_ctx
    ws = torch.zeros(bd.tts_decode_attn_workspace_size(w.B, w.q_len, w.Hq, w.Hkv, w.D, max_ctx),
                     dtype=torch.uint8, device="cuda")
    q = u.q if q is None else q
    out = torch.empty_like(q)
    bd.tts_decode_attn(cache, u.table, u.ctx_lens, max_ctx, q, out, ws, 1.0 / math.sqrt(w.D),
                       w.causal, err=err)
    torch.cuda.synchronize()
    return out, ws


def oracle_step_attn(orc, inp):
    w = inp["workload"]
    kp, vp = orc.kv_append(inp["k_pool"], inp["v_pool"], inp["block_table"], inp["ctx_before"],
                           inp["k_new"], inp["v_new"])
    out = orc.decode_attn(kp, vp, inp["block_table"], inp["ctx_lens"], inp["q"], inp["scale"], w.causal)
    return kp, vp, out


def check_attn(gpu_out, ref, dtype, label, parity=None):
    g = as_f64(host(gpu_out), dtype)
    assert np.isfinite(g).all(), f"{label}: non-finite attention output"
    bad, mx_abs, mx_rel = attn_errors(g, ref)
    if parity is not None:
        parity(f"attention {label}", max_abs=mx_abs, max_rel=mx_rel, elements=int(g.size))
    assert bad == 0, f"{label}: {bad} elements outside tolerance (max-abs {mx_abs})"
    # The absolute bound holds on every element (so reading the tolerance as
    # "absolute or relative" admits nothing more), and the relative bound
    # holds wherever it is the larger of the two.
    assert mx_abs <= ATOL, f"{label}: max-abs {mx_abs} above {ATOL}"
    rb = rel_where_binding(g, ref)
    assert rb <= RTOL, f"{label}: relative error {rb} above {RTOL} where |o| >= {ATOL / RTOL}"
    if dtype == "f32":
        assert mx_abs < 1e-4, f"{label}: fp32 attention error {mx_abs}"


# ------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_append_and_attention(orc, parity, wid):
    inp = wl.make_inputs(wid, with_head=False, with_verify=False)
    w = inp["workload"]
    u = Uploaded(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = gpu_append(u, err)
    out, ws = gpu_attn(u, cache, err=err)
    kp, vp, ref = oracle_step_attn(orc, inp)
    assert np.array_equal(host(u.k_pool).view(np.uint8), kp.view(np.uint8)), "K pool after append"
    assert np.array_equal(host(u.v_pool).view(np.uint8), vp.view(np.uint8)), "V pool after append"
    check_attn(out, ref, w.dtype, w.name, parity)
    assert int(err.item()) == 0
    # the ticket counters at the end of the workspace are back to zero
    ctr_bytes = -(-(w.B * w.Hkv * 4) // 256) * 256
    assert int(ws[ws.numel() - ctr_bytes:].count_nonzero()) == 0


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_head_select(orc, parity, wid):
    inp = wl.make_inputs(wid, with_verify=False)
    w = inp["workload"]
    u = Uploaded(inp)
    mode = bd.TTS_GUMBEL if w.mode == "gumbel" else bd.TTS_ARGMAX
    ids = torch.empty(w.R, dtype=torch.int32, device="cuda")
    best = torch.empty(w.R, dtype=torch.float32, device="cuda")
    ws = torch.zeros(bd.tts_head_workspace_size(w.R, w.V), dtype=torch.uint8, device="cuda")
    logits = torch.empty((w.R, w.V), dtype=torch.float32, device="cuda") if w.logits_out else None
    for rep in range(2):  # the workspace is reused as left by the first call
        bd.tts_codebook_head_select(u.h, u.W, ids, ws, mode=mode, temperature=w.T, seed=u.seed,
                                    step=u.step, best=best, logits_out=logits)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero()) == 0, "head workspace not left zeroed"
    rows = np.arange(w.R)  # every row
    ref = orc.head_select(np.ascontiguousarray(inp["h"][rows]), inp["W"], w.mode, w.T,
                          inp["seed"][rows], inp["step"][rows], want_logits=w.logits_out)
    got = host(ids)[rows]
    hard, ties = compare_ids(got, ref)
    parity(f"head {w.name}", rows=len(rows), near_ties=ties, hard=len(hard))
    assert not hard, f"ids differ outside near-ties at rows {hard[:10]}"
    fin = ref["best"] - ref["second"] >= NEAR_TIE
    assert np.allclose(host(best)[rows][fin], ref["best"][fin], rtol=1e-4, atol=1e-3)
    if logits is not None:
        gl = host(logits)[rows]
        assert np.allclose(gl, ref["logits"], rtol=1e-4, atol=1e-4), \
            f"logits max err {np.abs(gl - ref['logits']).max()}"


def test_spec_verify(orc, parity):
    inp = wl.make_inputs(5, with_head=False)
    w = inp["workload"]
    u = Uploaded(inp)
    for bonus in (False, True):
        n_acc = torch.empty(w.B, dtype=torch.int32, device="cuda")
        nxt = torch.empty(w.B, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        bd.tts_spec_verify(u.target_logits, u.draft_probs, u.draft_tokens, w.T, u.vseed, u.vstep,
                           n_acc, nxt, bonus=bonus, err=err)
        torch.cuda.synchronize()
        ref = orc.spec_verify(inp["target_logits"], inp["draft_probs"], inp["draft_tokens"], w.T,
                              inp["vseed"], inp["vstep"], bonus=bonus)
        tie = (ref["gap_accept"] < NEAR_TIE) | (ref["gap_resid"] < NEAR_TIE)
        bad = (host(n_acc) != ref["n_accepted"]) | (host(nxt) != ref["next_token"])
        parity(f"verify {w.name} bonus={int(bonus)}", streams=w.B, near_ties=int(tie.sum()),
               hard=int((bad & ~tie).sum()), accepted_mean=float(ref["n_accepted"].mean()))
        assert not (bad & ~tie).any(), f"verify differs at streams {np.nonzero(bad & ~tie)[0][:10]}"
        assert int(err.item()) == 0


def _verify_case(B, K, V, seed):
    """Seeded verify inputs of any shape: N(0,1) target logits, draft-model
    probabilities and tokens, per-stream Philox keys."""
    rng = np.random.default_rng(seed)
    tl = rng.standard_normal((B, K + 1, V), dtype=np.float32)
    dp, dt = wl.draft_model_outputs(B, K, V, rng)
    vseed = (wl.PHILOX_SEED_MUL * 11 + np.arange(B)).astype(np.uint64)
    vstep = np.full(B, 3, dtype=np.uint64)
    return tl, dp, dt, vseed, vstep


# Shapes around both verify kernels: shared-memory staged (small rows, ragged
# 16-byte ends, one to sixteen drafts) and streaming (rows too large to stage).
@pytest.mark.parametrize("B,K,V", [(8, 1, 37), (16, 3, 4097), (8, 7, 1000), (6, 16, 513), (4, 4, 16385),
                                   (3, 2, 3)])
def test_spec_verify_shapes(orc, B, K, V):
    tl, dp, dt, vseed, vstep = _verify_case(B, K, V, 1234 + B * K + V)
    T = 0.7
    for bonus in (False, True):
        n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        bd.tts_spec_verify(dev(tl), dev(dp), dev(dt), T, dev(vseed), dev(vstep), n_acc, nxt, bonus=bonus, err=err)
        torch.cuda.synchronize()
        ref = orc.spec_verify(tl, dp, dt, T, vseed, vstep, bonus=bonus)
        tie = (ref["gap_accept"] < NEAR_TIE) | (ref["gap_resid"] < NEAR_TIE)
        bad = (host(n_acc) != ref["n_accepted"]) | (host(nxt) != ref["next_token"])
        assert not (bad & ~tie).any(), f"verify B={B} K={K} V={V} bonus={bonus} differs at {np.nonzero(bad & ~tie)[0]}"
        assert int(err.item()) == 0


@pytest.mark.parametrize("V", [4097, 16385])
def test_spec_verify_zero_residual_draws_from_target(orc, V):
    """A residual that is zero everywhere: draft "probabilities" of 1 for every
    entry make max(p_t - p_d, 0) vanish, so a rejection draws from p_t itself
    (the fallback of the residual draw), in the staged kernel (V = 4097) and
    the streaming one (V = 16385); compared with the oracle."""
    B, K = 16, 4
    tl, _, dt, vseed, vstep = _verify_case(B, K, V, 4242 + V)
    dp = np.ones((B, K, V), dtype=np.float32)
    T = 0.7
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_spec_verify(dev(tl), dev(dp), dev(dt), T, dev(vseed), dev(vstep), n_acc, nxt, err=err)
    torch.cuda.synchronize()
    ref = orc.spec_verify(tl, dp, dt, T, vseed, vstep)
    assert (ref["n_accepted"] < K).all(), "every stream should reject somewhere (p_d = 1)"
    tie = (ref["gap_accept"] < NEAR_TIE) | (ref["gap_resid"] < NEAR_TIE)
    bad = (host(n_acc) != ref["n_accepted"]) | (host(nxt) != ref["next_token"])
    assert not (bad & ~tie).any(), f"differs at streams {np.nonzero(bad & ~tie)[0]}"
    assert (host(nxt) >= 0).all() and int(err.item()) == 0


def test_spec_verify_bad_token():
    """A draft token outside the vocabulary where the walk reaches it stops the
    walk there with no draw and sets the token error bit."""
    B, K, V = 4, 3, 4097
    tl, dp, dt, vseed, vstep = _verify_case(B, K, V, 77)
    dt = dt.copy()
    dt[1, 0] = V
    dt[2, 0] = -5
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_spec_verify(dev(tl), dev(dp), dev(dt), 0.7, dev(vseed), dev(vstep), n_acc, nxt, err=err)
    torch.cuda.synchronize()
    assert host(n_acc)[1] == 0 and host(nxt)[1] == -1
    assert host(n_acc)[2] == 0 and host(nxt)[2] == -1
    assert int(err.item()) & bd._lib.ERRBIT_TOKEN


@pytest.mark.parametrize("wid", [3, 5])
def test_full_step_chain(orc, parity, wid):
    """Append -> attention -> head on one stream, as the benchmark runs it."""
    inp = wl.make_inputs(wid, with_verify=False)
    w = inp["workload"]
    u = Uploaded(inp)
    cache = bd.KVCache(u.k_pool, u.v_pool)
    mode = bd.TTS_GUMBEL if w.mode == "gumbel" else bd.TTS_ARGMAX
    step = DecodeStep(cache, u.W, w.Hq, w.B, w.ctx_hi, q_len=w.q_len, causal=w.causal, mode=mode,
                      temperature=w.T)
    ids = step(u.table, u.ctx_before, u.ctx_lens, u.q, u.k_new, u.v_new, seed=u.seed, step=u.step)
    torch.cuda.synchronize()
    _, _, attn = oracle_step_attn(orc, inp)
    h = wl.f32_to_bf16(attn.reshape(w.R, w.Hq * w.D).astype(np.float32))
    rows = np.arange(w.R)  # every row
    ref = orc.head_select(np.ascontiguousarray(h[rows]), inp["W"], w.mode, w.T, inp["seed"][rows],
                          inp["step"][rows])
    hard, ties = compare_ids(host(ids)[rows], ref)
    parity(f"step chain {w.name}", rows=len(rows), near_ties=ties, hard=len(hard))
    assert not hard
    assert int(step.err.item()) == 0


# ------------------------------------------------------- small / edge shapes

SMALL = [
    # (base, B, Hq, Hkv, q_len, causal, ctx list, permute)
    (3, 1, 16, 8, 1, False, [1], True),
    (3, 4, 16, 8, 1, False, [15, 16, 17, 33], True),
    (3, 3, 16, 8, 1, False, [255, 256, 257], False),
    (3, 2, 16, 8, 1, False, [4096, 1], True),
    (5, 3, 16, 8, 5, True, [5, 6, 21], True),
    (5, 2, 16, 8, 5, True, [300, 17], False),
    (3, 3, 8, 8, 1, False, [40, 100, 7], True),     # MHA: one query row per KV head
    (3, 2, 16, 4, 1, False, [70, 9], True),          # group 4
    (3, 2, 8, 1, 2, True, [31, 64], True),           # group 8, q_len 2 -> 16 rows
    (1, 3, 4, 2, 1, False, [1, 16, 100], True),      # fp32
    (1, 2, 4, 2, 3, True, [3, 50], True),            # fp32 causal
]


@pytest.mark.parametrize("case", SMALL, ids=[f"s{i}" for i in range(len(SMALL))])
def test_small_shapes(orc, parity, case):
    base, B, Hq, Hkv, q_len, causal, ctx, permute = case
    w = wl.custom(base, B=B, Hq=Hq, Hkv=Hkv, q_len=q_len, causal=causal, ctx_lo=1,
                  ctx_hi=max(ctx), permute_table=permute)
    inp = wl.make_inputs(w, seed=99 + len(ctx), ctx_lens=ctx, with_head=False, with_verify=False)
    u = Uploaded(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = gpu_append(u, err)
    out, _ = gpu_attn(u, cache, err=err)
    _, _, ref = oracle_step_attn(orc, inp)
    check_attn(out, ref, w.dtype, f"small {case}", parity)
    assert int(err.item()) == 0


def test_context_bound_invariance(orc):
    """A looser max_ctx_len bound (a larger grid with more empty splits) changes nothing."""
    inp = wl.make_inputs(3, with_head=False, with_verify=False)
    u = Uploaded(inp)
    cache = gpu_append(u)
    a, _ = gpu_attn(u, cache)
    b, _ = gpu_attn(u, cache, max_ctx=4096)
    assert torch.equal(a, b)


def test_block_permutation_invariance():
    inp = wl.make_inputs(wl.custom(3, B=8), with_head=False, with_verify=False)
    u = Uploaded(inp)
    cache = gpu_append(u)
    a, _ = gpu_attn(u, cache)
    nb = inp["num_blocks"]
    perm = np.random.default_rng(3).permutation(nb)
    kp = np.empty_like(inp["k_pool"])
    vp = np.empty_like(inp["v_pool"])
    kp[perm] = host(u.k_pool)
    vp[perm] = host(u.v_pool)
    t2 = np.where(inp["block_table"] >= 0, perm[np.maximum(inp["block_table"], 0)], -1).astype(np.int32)
    u.k_pool, u.v_pool, u.table = dev(kp), dev(vp), dev(t2)
    b, _ = gpu_attn(u, bd.KVCache(u.k_pool, u.v_pool))
    assert torch.equal(a, b)


def test_batch_compaction(orc):
    """Dropping streams from the batch leaves the others' outputs unchanged up to
    rounding (the work split, and so the summation order, follows the batch)."""
    inp = wl.make_inputs(wl.custom(3, B=12), with_head=False, with_verify=False)
    u = Uploaded(inp)
    cache = gpu_append(u)
    full, _ = gpu_attn(u, cache)
    keep = np.array([0, 3, 4, 9, 11])
    u2 = Uploaded(dict(inp))
    u2.k_pool, u2.v_pool = u.k_pool, u.v_pool
    u2.w = wl.custom(3, B=len(keep))
    u2.table = dev(np.ascontiguousarray(inp["block_table"][keep]))
    u2.ctx_lens = dev(inp["ctx_lens"][keep])
    u2.q = dev(np.ascontiguousarray(inp["q"][keep]))
    part, _ = gpu_attn(u2, bd.KVCache(u2.k_pool, u2.v_pool))
    a = as_f64(host(part), "bf16")
    b = as_f64(host(full[torch.from_numpy(keep).cuda()]), "bf16")
    bad, mx_abs, _ = attn_errors(a, b)
    assert bad == 0 and mx_abs < 2e-2, f"compaction changed outputs by {mx_abs}"


# --------------------------------------------------- invalid data on device

def test_invalid_block_id_is_flagged_and_skipped(orc):
    w = wl.custom(3, B=3, ctx_lo=20, ctx_hi=80)
    inp = wl.make_inputs(w, seed=5, ctx_lens=[40, 80, 20], with_head=False, with_verify=False)
    u = Uploaded(inp)
    cache = gpu_append(u)
    bad = inp["block_table"].copy()
    bad[1, 2] = inp["num_blocks"] + 1000   # stream 1's third block points outside the pool
    u.table = dev(bad)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = gpu_attn(u, cache, err=err)
    assert int(err.item()) & bd._lib.ERRBIT_BLOCK_ID
    o = as_f64(host(out), "bf16")
    assert np.isfinite(o).all()
    _, _, ref = oracle_step_attn(orc, inp)
    for b in (0, 2):   # untouched streams still match
        assert attn_errors(o[b], ref[b])[0] == 0


def test_out_of_range_context_gives_zeros():
    w = wl.custom(3, B=2, ctx_lo=20, ctx_hi=64)
    inp = wl.make_inputs(w, seed=6, ctx_lens=[30, 64], with_head=False, with_verify=False)
    u = Uploaded(inp)
    cache = gpu_append(u)
    u.ctx_lens = dev(np.array([30, 65], dtype=np.int32))  # beyond max_ctx_len = 64
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = gpu_attn(u, cache, max_ctx=64, err=err)
    assert int(err.item()) & bd._lib.ERRBIT_CTX_LEN
    assert int(out[1].float().abs().sum().item()) == 0
    assert torch.isfinite(out.float()).all()


def test_draft_token_outside_vocab_is_flagged():
    w = wl.custom(5, B=4, V=97, H=64)
    inp = wl.make_inputs(w, seed=2, with_head=False)
    inp["draft_tokens"][2, 0] = 97
    u = Uploaded(inp)
    n_acc = torch.empty(4, dtype=torch.int32, device="cuda")
    nxt = torch.empty(4, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_spec_verify(u.target_logits, u.draft_probs, u.draft_tokens, w.T, u.vseed, u.vstep,
                       n_acc, nxt, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & bd._lib.ERRBIT_TOKEN
    assert int(nxt[2].item()) == -1 and int(n_acc[2].item()) == 0


# ------------------------------------------------------------ head shapes

HEAD_SHAPES = [(1, 64, 300), (17, 128, 1000), (256, 64, 129), (257, 64, 200), (320, 128, 257),
               (5, 2048, 4097),
               (3, 64, 1),      # one entry: rows whose boundary is masked choose nothing (-1)
               (9, 64, 7),      # fewer entries than one 8-entry selection group
               (4096, 64, 64)]  # the largest batch: 16 chunks of 256 rows


@pytest.mark.parametrize("R,H,V", HEAD_SHAPES)
@pytest.mark.parametrize("mode", ["argmax", "gumbel"])
def test_head_shapes(orc, R, H, V, mode):
    rng = np.random.default_rng(R * 7 + V)
    h = wl.f32_to_bf16(rng.standard_normal((R, H), dtype=np.float32))
    W = wl.f32_to_bf16(0.05 * rng.standard_normal((V, H), dtype=np.float32))
    seed = np.arange(R, dtype=np.uint64) + 77
    step = np.full(R, 3, dtype=np.uint64)
    eos = (np.arange(R) % 3 != 0).astype(np.uint8)
    ids = torch.empty(R, dtype=torch.int32, device="cuda")
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    ws = torch.zeros(bd.tts_head_workspace_size(R, V), dtype=torch.uint8, device="cuda")
    m = bd.TTS_GUMBEL if mode == "gumbel" else bd.TTS_ARGMAX
    bd.tts_codebook_head_select(dev(h), dev(W), ids, ws, mode=m, temperature=0.8, seed=dev(seed),
                                step=dev(step), eos_allowed=dev(eos), logits_out=logits)
    torch.cuda.synchronize()
    ref = orc.head_select(h, W, mode, 0.8, seed, step, eos_allowed=eos, want_logits=True)
    assert np.allclose(host(logits), ref["logits"], rtol=1e-4, atol=1e-4)
    gids = host(ids)
    none = ref["ids"] < 0                       # every entry masked: no choice either side
    assert np.array_equal(gids[none], ref["ids"][none])
    hard, ties = compare_ids(np.where(none, 0, gids), {k: np.where(none, 0, v) if k == "ids" else
                                                       np.where(none, 1.0, v) if k == "best" else
                                                       np.where(none, 0.0, v) for k, v in ref.items()
                                                       if k in ("ids", "best", "second")})
    assert not hard, f"rows {hard[:10]}"
    assert int(ws.count_nonzero()) == 0


# Shapes of the split build (at most 64 rows, no logits written, vocab tiles
# all in one wave): one to 64 rows, hidden widths 256 to 4096 (4- and 8-CTA
# cluster splits), ragged and exact vocab tiles, fewer entries than one
# selection group, a single entry.
SPLIT_SHAPES = [(1, 256, 300), (16, 2048, 4097), (17, 512, 1000), (33, 1024, 2049), (64, 2048, 4097),
                (64, 2048, 129), (48, 4096, 513), (5, 256, 7), (3, 256, 1), (64, 256, 4224)]


@pytest.mark.parametrize("R,H,V", SPLIT_SHAPES)
@pytest.mark.parametrize("mode", ["argmax", "gumbel"])
def test_head_split_shapes(orc, parity, R, H, V, mode):
    rng = np.random.default_rng(R * 11 + V + H)
    h = wl.f32_to_bf16(rng.standard_normal((R, H), dtype=np.float32))
    W = wl.f32_to_bf16((0.5 / math.sqrt(H)) * rng.standard_normal((V, H), dtype=np.float32))
    seed = np.arange(R, dtype=np.uint64) + 501
    step = np.full(R, 9, dtype=np.uint64)
    eos = (np.arange(R) % 4 != 1).astype(np.uint8)
    ids = torch.empty(R, dtype=torch.int32, device="cuda")
    best = torch.empty(R, dtype=torch.float32, device="cuda")
    ws = torch.zeros(bd.tts_head_workspace_size(R, V), dtype=torch.uint8, device="cuda")
    m = bd.TTS_GUMBEL if mode == "gumbel" else bd.TTS_ARGMAX
    ref = orc.head_select(h, W, mode, 0.9, seed, step, eos_allowed=eos)
    for rep in range(2):  # the workspace as the first call left it
        ids.fill_(-9)
        bd.tts_codebook_head_select(dev(h), dev(W), ids, ws, mode=m, temperature=0.9, seed=dev(seed),
                                    step=dev(step), eos_allowed=dev(eos), best=best)
        torch.cuda.synchronize()
        gids = host(ids)
        none = ref["ids"] < 0
        assert np.array_equal(gids[none], ref["ids"][none])
        hard, ties = compare_ids(np.where(none, 0, gids), {k: np.where(none, 0, v) if k == "ids" else
                                                           np.where(none, 1.0, v) if k == "best" else
                                                           np.where(none, 0.0, v) for k, v in ref.items()})
        assert not hard, f"rows {hard[:10]}"
        fin = ~none & (ref["best"] - ref["second"] >= NEAR_TIE)
        assert np.allclose(host(best)[fin], ref["best"][fin], rtol=1e-4, atol=1e-3)
        assert int(ws.count_nonzero()) == 0
    parity(f"split head R{R} H{H} V{V} {mode}", near_ties=ties, hard=len(hard))


def test_head_boundary_token_mask(orc):
    R, H, V = 8, 64, 513
    h = wl.f32_to_bf16(np.ones((R, H), dtype=np.float32))
    Wf = np.zeros((V, H), dtype=np.float32)
    Wf[V - 1] = 1.0
    Wf[100] = 0.5
    W = wl.f32_to_bf16(Wf)
    eos = np.array([1, 0] * 4, dtype=np.uint8)
    ids = torch.empty(R, dtype=torch.int32, device="cuda")
    ws = torch.zeros(bd.tts_head_workspace_size(R, V), dtype=torch.uint8, device="cuda")
    bd.tts_codebook_head_select(dev(h), dev(W), ids, ws, eos_allowed=dev(eos))
    torch.cuda.synchronize()
    assert list(host(ids)) == [V - 1, 100] * 4


def test_graphed_step_matches_direct_step(orc, parity):
    """The captured serving step (host copies in, step, ids out) gives the same
    ids as the direct step, and both match the oracle: its attention on the
    same inputs, its head on the step's own attention output."""
    inp = wl.make_inputs(wl.custom(3, B=24), with_verify=False)
    w = inp["workload"]
    u = Uploaded(inp)
    cache = bd.KVCache(u.k_pool, u.v_pool)
    step = DecodeStep(cache, u.W, w.Hq, w.B, w.ctx_hi)
    direct = step(u.table, u.ctx_before, u.ctx_lens, u.q, u.k_new, u.v_new).clone()
    g = GraphedStep(step, {"block_table": u.table, "ctx_before": u.ctx_before, "ctx_lens": u.ctx_lens,
                           "q": u.q, "k_new": u.k_new, "v_new": u.v_new})
    for _ in range(3):
        g.ids_host.fill_(-7)           # a replay that did not finish would leave this
        assert torch.equal(g().clone(), direct.cpu())
    # the captured step against the oracle directly
    _, _, ref_attn = oracle_step_attn(orc, inp)
    check_attn(step.out, ref_attn, w.dtype, "captured step custom-b24", parity)
    h = host(step.out).reshape(w.R, -1)
    ref = orc.head_select(h, inp["W"])
    hard, ties = compare_ids(g.ids_host.numpy().copy(), ref)
    parity("captured step custom-b24 head", rows=w.R, near_ties=ties, hard=len(hard))
    assert not hard, f"captured step ids differ from the oracle at rows {hard}"
    # new inputs written into the pinned host views reach the step
    q2 = torch.randn(u.q.shape, device="cuda").to(u.q.dtype)
    direct2 = step(u.table, u.ctx_before, u.ctx_lens, q2, u.k_new, u.v_new).clone()
    g.host["q"].copy_(q2.cpu())
    g.ids_host.fill_(-7)
    assert torch.equal(g().clone(), direct2.cpu())
    assert not torch.equal(direct2, direct)
    assert g.boundary_count == int((direct2 == w.V - 1).sum())
    assert int(step.err.item()) == 0


def test_graphed_step_run_returns_each_launchs_ids():
    """tts_step_graph_run returns once that launch's ids are in host memory:
    the query rows alternate between two sets, the ids are copied the moment
    the call returns, and the launch numbering starts past two asynchronous
    launches."""
    inp = wl.make_inputs(wl.custom(3, B=24), with_verify=False)
    w = inp["workload"]
    u = Uploaded(inp)
    cache = bd.KVCache(u.k_pool, u.v_pool)
    step = DecodeStep(cache, u.W, w.Hq, w.B, w.ctx_hi)
    qs = [u.q, torch.randn(u.q.shape, device="cuda").to(u.q.dtype)]
    want = [step(u.table, u.ctx_before, u.ctx_lens, q, u.k_new, u.v_new).cpu().clone() for q in qs]
    assert not torch.equal(want[0], want[1])
    g = GraphedStep(step, {"block_table": u.table, "ctx_before": u.ctx_before, "ctx_lens": u.ctx_lens,
                           "q": u.q, "k_new": u.k_new, "v_new": u.v_new})
    g.graph.launch(g.stream)
    g.graph.launch(g.stream)
    g.stream.synchronize()
    for i in range(20):
        g.host["q"].copy_(qs[i & 1].cpu())
        g.ids_host.fill_(-7)
        assert torch.equal(g().clone(), want[i & 1]), f"run {i} returned before its ids"
    assert int(step.err.item()) == 0


def test_graphed_step_boundary_count():
    """The captured step counts the rows whose id is the boundary token V - 1
    on the device: a boundary row of W aligned with half the streams'
    attention outputs makes exactly those streams end."""
    inp = wl.make_inputs(wl.custom(3, B=32), with_verify=False)
    w = inp["workload"]
    u = Uploaded(inp)
    cache = bd.KVCache(u.k_pool, u.v_pool)
    W = u.W.clone()
    step = DecodeStep(cache, W, w.Hq, w.B, w.ctx_hi)
    step(u.table, u.ctx_before, u.ctx_lens, u.q, u.k_new, u.v_new)  # fills the attention output
    out = step.out.view(w.B, -1).float()
    # boundary row: a large multiple of stream 0..15's mean output direction
    direction = out[:16].mean(0)
    W[w.V - 1] = (50.0 * direction / direction.norm()).to(W.dtype)
    step.W = W
    direct = step(u.table, u.ctx_before, u.ctx_lens, u.q, u.k_new, u.v_new).clone()
    expect = int((direct == w.V - 1).sum())
    assert expect > 0
    g = GraphedStep(step, {"block_table": u.table, "ctx_before": u.ctx_before, "ctx_lens": u.ctx_lens,
                           "q": u.q, "k_new": u.k_new, "v_new": u.v_new})
    ids = g().clone()
    assert torch.equal(ids, direct.cpu())
    assert g.boundary_count == expect
