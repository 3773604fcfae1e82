"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each `check_*` takes an `oracle.Oracle` and raises AssertionError when the
oracle disagrees with a closed form, a library routine (numpy's Philox4x64-10,
numpy matmul, torch's scaled_dot_product_attention, scipy's distributions), an
invariance of the method, or a distributional theorem.  The pages print no
numeric worked example for this path, so these are the pins.

`tests/test_oracle_pins.py` runs every check on the real oracle;
`tests/test_oracle_mutants.py` plants plausible mistakes in copies of the
oracle source and requires each mistake to fail at least one check.
"""
from __future__ import annotations

import math
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import workloads as wl  # noqa: E402

EULER_GAMMA = 0.5772156649015329
U64 = 1 << 64


# ------------------------------------------------------------------ helpers

def _numpy_philox_block(ctr, key):
    """The four 64-bit words numpy's Philox4x64-10 produces for counter `ctr`.

    numpy advances its 256-bit counter before each block, so its state is set
    to ctr - 1 (with borrow)."""
    c = [int(x) for x in ctr]
    value = sum(x << (64 * i) for i, x in enumerate(c)) - 1
    value %= 1 << 256
    state = [(value >> (64 * i)) & (U64 - 1) for i in range(4)]
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=np.array(state, dtype=np.uint64))
    return [int(x) for x in bg.random_raw(4)]


def _chi2_p(observed, probs):
    from scipy.stats import chisquare
    observed = np.asarray(observed, dtype=np.float64)
    expected = np.asarray(probs, dtype=np.float64) * observed.sum()
    keep = expected > 0
    assert observed[~keep].sum() == 0, "mass on a zero-probability outcome"
    return chisquare(observed[keep], expected[keep]).pvalue


def _softmax64(x, T=1.0):
    x = np.asarray(x, dtype=np.float64) / T
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def attn_case(seed, B, Hq, Hkv, D, q_len, ctx_lens, dtype="f32", permute=False):
    """Pools holding every context token (including this step's), q, table."""
    rng = np.random.default_rng(seed)
    L = np.asarray(ctx_lens, dtype=np.int32)
    max_blocks = int(-(-L.max() // wl.BLOCK))
    num_blocks, table = wl.layout_blocks(L, max_blocks, spare=2, permute=permute, rng=rng)
    kp = wl.fill_pool(num_blocks, Hkv, D, dtype, table, L, rng)
    vp = wl.fill_pool(num_blocks, Hkv, D, dtype, table, L, rng)
    q = wl._store(rng.standard_normal((B, q_len, Hq, D), dtype=np.float32), dtype)
    return dict(k_pool=kp, v_pool=vp, block_table=table, ctx_lens=L, q=q)


def gather(pool, table, b, L, dtype):
    """Logical [L][Hkv][D] float64 view of stream b's cache."""
    t = np.arange(L)
    blocks = table[b, t // wl.BLOCK]
    return wl.to_f32(pool[blocks, :, t % wl.BLOCK, :], dtype).astype(np.float64)


# ------------------------------------------------------------------- Philox

def check_philox_matches_numpy(o):
    keys = [(1, 2), (0, 0), (U64 - 1, 12345), (7919 * 4 + 17, 3)]
    ctrs = [(1, 0, 0, 0), (0, 0, 0, 0), (5, 1, 0, 0), (U64 - 1, 2, 3, 0), (123456, 0, 4, 0),
            (9, 1, 2, 3)]
    for key in keys:
        for ctr in ctrs:
            got = [int(x) for x in o.philox(ctr, key)]
            want = _numpy_philox_block(ctr, key)
            assert got == want, f"Philox4x64-10 mismatch at ctr={ctr} key={key}"


def check_uniform_words(o):
    """Uniform idx takes half (idx % 8) of the block at counter (idx // 8, tag, pos, 0),
    low half first, and maps its top 23 bits k to (2k + 1) / 2^24."""
    for (seed, step, tag, pos) in [(3, 0, 0, 0), (99, 7, 1, 0), (5, 5, 2, 3)]:
        for idx in [0, 1, 2, 5, 7, 8, 13, 4096, 16384]:
            words = _numpy_philox_block((idx // 8, tag, pos, 0), (seed, step))
            w = words[(idx % 8) // 2]
            half = (w >> 32) if idx % 2 else (w & 0xFFFFFFFF)
            want = (2 * (half >> 9) + 1) / 2.0 ** 24
            got = o.uniform(seed, step, tag, pos, idx)
            assert got == want, f"uniform({seed},{step},{tag},{pos},{idx}) = {got}, want {want}"
            assert 0.0 < got < 1.0


def check_gumbel_distribution(o):
    from scipy.stats import kstest
    g = np.array([o.gumbel(11, 3, 0, 0, i) for i in range(20000)])
    assert abs(g.mean() - EULER_GAMMA) < 0.03, g.mean()
    assert abs(g.var() - math.pi ** 2 / 6) < 0.08, g.var()
    assert kstest(g, "gumbel_r").pvalue > 1e-4


# --------------------------------------------------------------- attention

def check_attn_matches_sdpa(o):
    """torch's scaled_dot_product_attention on the gathered cache (float64)."""
    import torch
    import torch.nn.functional as F
    for (Hq, Hkv, D, q_len, causal, L, dtype, seed) in [
            (4, 2, 64, 1, False, [17, 1, 40], "f32", 1),
            (8, 2, 32, 3, True, [3, 33, 20], "bf16", 2),
            (6, 6, 16, 5, True, [5, 16, 48], "f32", 3),
            (4, 1, 16, 2, False, [9, 31], "bf16", 4)]:
        c = attn_case(seed, len(L), Hq, Hkv, D, q_len, L, dtype, permute=True)
        scale = 0.7 / math.sqrt(D)
        out = o.decode_attn(c["k_pool"], c["v_pool"], c["block_table"], c["ctx_lens"], c["q"],
                            scale, causal)
        g = Hq // Hkv
        for b, Lb in enumerate(L):
            k = torch.from_numpy(gather(c["k_pool"], c["block_table"], b, Lb, dtype))
            v = torch.from_numpy(gather(c["v_pool"], c["block_table"], b, Lb, dtype))
            k = k.permute(1, 0, 2).repeat_interleave(g, dim=0)
            v = v.permute(1, 0, 2).repeat_interleave(g, dim=0)
            q = torch.from_numpy(wl.to_f32(c["q"][b], dtype).astype(np.float64)).permute(1, 0, 2)
            mask = None
            if causal:
                t = torch.arange(Lb)[None, :]
                j = torch.arange(q_len)[:, None]
                mask = t < (Lb - q_len + j + 1)
            ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
            got = torch.from_numpy(out[b]).permute(1, 0, 2)
            err = (got - ref).abs().max().item()
            assert err < 1e-10, f"attention vs SDPA: {err}"


def check_attn_constant_keys(o):
    """Equal scores give the mean of the visible values."""
    for (q_len, causal, L) in [(1, False, [1, 16, 37]), (5, True, [5, 21, 64])]:
        c = attn_case(7, len(L), 4, 2, 64, q_len, L)
        kp = c["k_pool"]
        kp[:] = np.float32(0.25)
        out = o.decode_attn(kp, c["v_pool"], c["block_table"], c["ctx_lens"], c["q"], 0.125, causal)
        for b, Lb in enumerate(L):
            v = gather(c["v_pool"], c["block_table"], b, Lb, "f32")
            for j in range(q_len):
                lim = Lb - q_len + j + 1 if causal else Lb
                for h in range(4):
                    want = v[:lim, h // 2, :].mean(axis=0)
                    assert np.allclose(out[b, j, h], want, atol=1e-12), "constant keys"


def check_attn_dominant_score(o):
    """One key aligned with the query and scaled up takes all the weight."""
    L = [30, 45]
    c = attn_case(8, 2, 2, 1, 16, 1, L)
    kp, table, q = c["k_pool"], c["block_table"], c["q"]
    picks = [3, 44]
    for b, t in enumerate(picks):
        kp[table[b, t // 16], 0, t % 16, :] = 400.0 * q[b, 0, 0, :]
        q[b, 0, 1, :] = q[b, 0, 0, :]
    out = o.decode_attn(kp, c["v_pool"], table, c["ctx_lens"], q, 1.0, False)
    for b, t in enumerate(picks):
        v = gather(c["v_pool"], table, b, L[b], "f32")[t, 0]
        for h in range(2):
            assert np.allclose(out[b, 0, h], v, atol=1e-9), "dominant score"


def check_attn_single_token(o):
    c = attn_case(9, 3, 4, 4, 32, 1, [1, 1, 1])
    out = o.decode_attn(c["k_pool"], c["v_pool"], c["block_table"], c["ctx_lens"], c["q"], 0.3)
    for b in range(3):
        v = gather(c["v_pool"], c["block_table"], b, 1, "f32")[0]
        assert np.array_equal(out[b, 0], v), "context of one token returns its value"


def check_attn_block_permutation(o):
    """Where blocks sit in the pool does not change the result."""
    L = [40, 7, 64]
    c = attn_case(10, 3, 4, 2, 64, 1, L, "bf16")
    nb = c["k_pool"].shape[0]
    perm = np.random.default_rng(1).permutation(nb)   # new position of each block
    kp2 = np.empty_like(c["k_pool"])
    vp2 = np.empty_like(c["v_pool"])
    kp2[perm] = c["k_pool"]
    vp2[perm] = c["v_pool"]
    t2 = np.where(c["block_table"] >= 0, perm[c["block_table"]], -1).astype(np.int32)
    a = o.decode_attn(c["k_pool"], c["v_pool"], c["block_table"], c["ctx_lens"], c["q"], 0.125)
    b = o.decode_attn(kp2, vp2, t2, c["ctx_lens"], c["q"], 0.125)
    assert np.array_equal(a, b), "block permutation changed the output"


def check_attn_verify_rows(o):
    """Row j of a causal q_len-row block equals a single-row step on the first
    ctx - q_len + j + 1 tokens."""
    L = [9, 33]
    q_len = 5
    c = attn_case(11, 2, 4, 2, 64, q_len, L, "bf16")
    full = o.decode_attn(c["k_pool"], c["v_pool"], c["block_table"], c["ctx_lens"], c["q"],
                         0.125, True)
    for j in range(q_len):
        Lj = np.array([x - q_len + j + 1 for x in L], dtype=np.int32)
        one = o.decode_attn(c["k_pool"], c["v_pool"], c["block_table"], Lj,
                            np.ascontiguousarray(c["q"][:, j:j + 1]), 0.125, False)
        assert np.allclose(full[:, j], one[:, 0], atol=1e-13), f"verify row {j}"


def check_kv_append_roundtrip(o):
    """Appended rows read back at their logical slots; every other slot is untouched."""
    w = wl.custom(1, B=3, q_len=5, ctx_lo=5, ctx_hi=40, permute_table=True, dtype="bf16")
    inp = wl.make_inputs(w, seed=5, with_head=False, with_verify=False)
    kp, vp = o.kv_append(inp["k_pool"], inp["v_pool"], inp["block_table"], inp["ctx_before"],
                         inp["k_new"], inp["v_new"])
    table = inp["block_table"]
    touched = np.zeros(kp.shape[0] * 16, dtype=bool)
    for b in range(w.B):
        for j in range(w.q_len):
            s = int(inp["ctx_before"][b]) + j
            blk = table[b, s // 16]
            assert np.array_equal(kp[blk, :, s % 16], inp["k_new"][b, j])
            assert np.array_equal(vp[blk, :, s % 16], inp["v_new"][b, j])
            touched[blk * 16 + s % 16] = True
    flat = lambda p: p.transpose(0, 2, 1, 3).reshape(kp.shape[0] * 16, -1)  # noqa: E731
    assert np.array_equal(flat(kp)[~touched], flat(inp["k_pool"])[~touched])
    assert np.array_equal(flat(vp)[~touched], flat(inp["v_pool"])[~touched])


# -------------------------------------------------------------------- head

def check_head_logits_match_matmul(o):
    rng = np.random.default_rng(12)
    for dtype in ("f32", "bf16"):
        h = wl._store(rng.standard_normal((5, 96), dtype=np.float32), dtype)
        W = wl._store(0.05 * rng.standard_normal((37, 96), dtype=np.float32), dtype)
        r = o.head_select(h, W, want_logits=True)
        ref = (wl.to_f32(h, dtype).astype(np.float64) @ wl.to_f32(W, dtype).astype(np.float64).T)
        assert np.allclose(r["logits"], ref.astype(np.float32), rtol=1e-6, atol=1e-7), "h W^T"
        assert np.array_equal(r["ids"], ref.argmax(axis=1)), "argmax of the logits"


def check_head_one_hot(o):
    """A one-hot hidden state picks one column of W, exactly."""
    rng = np.random.default_rng(13)
    W = rng.standard_normal((50, 8), dtype=np.float32)
    h = np.zeros((8, 8), dtype=np.float32)
    h[np.arange(8), np.arange(8)] = 1.0
    r = o.head_select(h, W, want_logits=True)
    assert np.array_equal(r["logits"], W.T), "one-hot rows select columns of W"


def check_head_constructed_winner(o):
    rng = np.random.default_rng(14)
    h = rng.standard_normal((6, 64), dtype=np.float32)
    W = 0.01 * rng.standard_normal((300, 64), dtype=np.float32)
    winners = [0, 17, 299, 150, 42, 298]
    for r, v in enumerate(winners):
        W[v] = 0.5 * h[r]
    got = o.head_select(h, W)["ids"]
    assert list(got) == winners, "constructed winner"


def check_head_ties_and_eos(o):
    V = 9
    W = np.ones((V, 4), dtype=np.float32)
    h = np.ones((3, 4), dtype=np.float32)
    r = o.head_select(h, W, eos_allowed=np.array([1, 0, 1], dtype=np.uint8))
    assert list(r["ids"]) == [0, 0, 0], "equal logits resolve to the lowest index"
    assert list(r["second"] - r["best"]) == [0, 0, 0]
    W2 = np.zeros((V, 4), dtype=np.float32)
    W2[V - 1] = 1.0
    W2[3] = 0.5
    r = o.head_select(h, W2, eos_allowed=np.array([1, 0, 1], dtype=np.uint8))
    assert list(r["ids"]) == [V - 1, 3, V - 1], "eos mask removes only the boundary token"


def _gumbel_freq(o, logits, T, rows, seed0=1000, step=0):
    logits = np.asarray(logits, dtype=np.float32)
    h = np.ones((rows, 1), dtype=np.float32)
    W = logits[:, None].copy()
    seed = np.arange(seed0, seed0 + rows, dtype=np.uint64)
    stp = np.full(rows, step, dtype=np.uint64)
    ids = o.head_select(h, W, mode="gumbel", T=T, seed=seed, step=stp)["ids"]
    return np.bincount(ids, minlength=len(logits))


def check_head_gumbel_is_softmax_draw(o):
    logits = [0.0, 0.9, 1.4, -0.6, 0.3]
    for T, step in [(0.7, 0), (1.6, 5)]:
        counts = _gumbel_freq(o, logits, T, 20000, step=step)
        p = _chi2_p(counts, _softmax64(logits, T))
        assert p > 1e-4, f"Gumbel draws do not follow softmax(logits/T) at T={T}: p={p}"


def check_head_gumbel_low_temperature(o):
    counts = _gumbel_freq(o, [0.1, 0.5, 0.45, -1.0], 1e-4, 500)
    assert counts[1] == 500, "T -> 0 reduces to argmax"


# ------------------------------------------------------------------ verify

def _verify_one(o, tl_rows, dp_rows, tokens, seeds, T=0.7, bonus=False):
    """Run the oracle over many independent streams that share logits."""
    B = len(seeds)
    K = len(dp_rows)
    tl = np.broadcast_to(np.asarray(tl_rows, dtype=np.float32), (B, K + 1, len(tl_rows[0])))
    dp = np.broadcast_to(np.asarray(dp_rows, dtype=np.float32), (B, K, len(tl_rows[0])))
    seed = np.asarray(seeds, dtype=np.uint64)
    return o.spec_verify(np.ascontiguousarray(tl), np.ascontiguousarray(dp),
                         np.ascontiguousarray(tokens, dtype=np.int32), T, seed,
                         np.zeros(B, dtype=np.uint64), bonus=bonus)


def check_verify_matching_draft_accepts_all(o):
    tl = np.random.default_rng(15).standard_normal((5, 33)).astype(np.float32)
    T = 0.7
    dp = _softmax64(tl[:4], T).astype(np.float32)
    tokens = np.tile(np.array([3, 0, 32, 7], dtype=np.int32), (50, 1))
    r = _verify_one(o, tl, dp, tokens, range(50), T)
    assert (r["n_accepted"] == 4).all() and (r["next_token"] == -1).all(), "p_d == p_t accepts all"


def check_verify_zero_target_rejects(o):
    rng = np.random.default_rng(16)
    tl = rng.standard_normal((5, 12)).astype(np.float32)
    tl[2, 6] = -1e30                      # p_t = 0 at draft 2's token
    dp = _softmax64(tl[:4], 0.7).astype(np.float32)
    dp[2] = _softmax64(rng.standard_normal(12))
    tokens = np.tile(np.array([1, 4, 6, 2], dtype=np.int32), (40, 1))
    r = _verify_one(o, tl, dp, tokens, range(40))
    assert (r["n_accepted"] == 2).all(), "a token the target gives zero mass is rejected"
    assert (r["next_token"] != 6).all() and (r["next_token"] >= 0).all()


def check_verify_zero_draft_rejects(o):
    tl = np.zeros((2, 6), dtype=np.float32)
    dp = np.array([[0.0, 0.2, 0.2, 0.2, 0.2, 0.2]], dtype=np.float32)
    tokens = np.zeros((30, 1), dtype=np.int32)
    r = _verify_one(o, tl, dp, tokens, range(30))
    assert (r["n_accepted"] == 0).all(), "p_d == 0 rejects"
    assert (r["next_token"] == 0).all(), "the residual then sits on the rejected token"


def check_verify_accept_rate(o):
    """P(accept) = min(1, p_t/p_d) at the drafted token."""
    tl = np.log(np.array([[0.2, 0.3, 0.5], [1, 1, 1]], dtype=np.float64)).astype(np.float32)
    dp = np.array([[0.5, 0.3, 0.2]], dtype=np.float32)
    n = 20000
    r = _verify_one(o, tl, dp, np.zeros((n, 1), dtype=np.int32), range(n), T=1.0)
    rate = r["n_accepted"].mean()
    ratio = 0.2 / 0.5
    assert abs(rate - ratio) < 5 * math.sqrt(ratio * (1 - ratio) / n), f"accept rate {rate}"


def check_verify_output_is_target_distribution(o):
    """Speculative sampling theorem: the first emitted token follows p_t."""
    rng = np.random.default_rng(17)
    T = 0.7
    tl = np.array([[1.0, 0.0, -1.0, 0.5], [0, 0, 0, 0]], dtype=np.float32)
    pd = np.array([[0.1, 0.6, 0.2, 0.1]], dtype=np.float32)
    n = 30000
    pd64 = pd[0].astype(np.float64)
    tokens = rng.choice(4, size=(n, 1), p=pd64 / pd64.sum()).astype(np.int32)
    r = _verify_one(o, tl, pd, tokens, range(5000, 5000 + n), T)
    emitted = np.where(r["n_accepted"] == 1, tokens[:, 0], r["next_token"])
    p = _chi2_p(np.bincount(emitted, minlength=4), _softmax64(tl[0], T))
    assert p > 1e-4, f"emitted tokens do not follow p_t: p={p}"


def check_verify_residual_distribution(o):
    T = 0.7
    tl = np.array([[1.0, 0.0, -1e30, 0.5, -0.5], [0] * 5], dtype=np.float32)
    pd = np.array([[0.1, 0.05, 0.1, 0.1, 0.65]], dtype=np.float32)
    n = 20000
    r = _verify_one(o, tl, pd, np.full((n, 1), 2, dtype=np.int32), range(n), T)
    assert (r["n_accepted"] == 0).all()
    pt = _softmax64(tl[0], T)
    res = np.maximum(pt - pd[0], 0.0)
    p = _chi2_p(np.bincount(r["next_token"], minlength=5), res / res.sum())
    assert p > 1e-4, f"replacement tokens do not follow the clamped residual: p={p}"


def check_verify_stops_at_first_rejection(o):
    rng = np.random.default_rng(18)
    T = 0.7
    tl = rng.standard_normal((5, 10)).astype(np.float32)
    tl[1, 3] = -1e30
    dp = _softmax64(tl[:4], T).astype(np.float32)
    tokens = np.tile(np.array([5, 3, 5, 5], dtype=np.int32), (20, 1))
    r = _verify_one(o, tl, dp, tokens, range(20), T)
    assert (r["n_accepted"] == 1).all(), "verification stops at the first rejection"


def check_verify_bonus_token(o):
    T = 0.7
    tl = np.array([[0.0, 0.0, 0.0], [0.2, -0.4, 1.1]], dtype=np.float32)
    dp = _softmax64(tl[:1], T).astype(np.float32)
    n = 20000
    tokens = np.zeros((n, 1), dtype=np.int32)
    r = _verify_one(o, tl, dp, tokens, range(n), T, bonus=True)
    assert (r["n_accepted"] == 1).all()
    p = _chi2_p(np.bincount(r["next_token"], minlength=3), _softmax64(tl[1], T))
    assert p > 1e-4, f"bonus token does not follow softmax(target[K]/T): p={p}"
    r = _verify_one(o, tl, dp, tokens[:10], range(10), T, bonus=False)
    assert (r["next_token"] == -1).all(), "no bonus token unless asked for"


def check_verify_draw_noise(o):
    """The replacement and bonus draws are Gumbel-max with the noise at
    counter position 0 of tag 2, whichever row they draw from: the token
    maximises log(residual) + G (or target / T + G for the bonus), G the
    pinned Philox-Gumbel of (seed, step, tag 2, position 0, entry).  Rows 1 and
    K = 2 are drawn from, so noise keyed by the row would differ."""
    T = 0.7
    V = 40
    rng = np.random.default_rng(19)
    tl = rng.standard_normal((3, V)).astype(np.float32)
    tl[1, 7] = -1e30                                   # p_t = 0 at draft 1's token: rejected
    dp = np.stack([_softmax64(tl[0], T), _softmax64(rng.standard_normal(V), 1.0)]).astype(np.float32)
    tokens = np.array([[3, 7]], dtype=np.int32)        # draft 0: p_d = p_t, accepted
    tlb = rng.standard_normal((3, V)).astype(np.float32)
    dpb = _softmax64(tlb[:2], T).astype(np.float32)    # every draft accepted: the bonus row 2 is drawn
    tokens_b = np.array([[1, 2]], dtype=np.int32)
    resid = np.maximum(_softmax64(tl[1], T) - dp[1].astype(np.float64), 0.0)
    checked = [0, 0]
    for seed in range(40):
        g = np.array([o.gumbel(seed, 0, 2, 0, v) for v in range(V)])
        for case, (x, d, tok, bonus) in enumerate(((tl, dp, tokens, False), (tlb, dpb, tokens_b, True))):
            r = _verify_one(o, x, d, tok, [seed], T, bonus=bonus)
            if case == 0:
                assert r["n_accepted"][0] == 1
                key = np.where(resid > 0, np.log(np.where(resid > 0, resid, 1.0)) + g, -np.inf)
            else:
                if r["n_accepted"][0] != 2:
                    continue
                key = x[2].astype(np.float64) / T + g
            top = np.sort(key)[-2:]
            if top[1] - top[0] < 1e-3:
                continue
            assert r["next_token"][0] == int(np.argmax(key)), f"seed {seed}: {'bonus' if bonus else 'residual'} draw"
            checked[case] += 1
    assert min(checked) >= 30, checked


# ---------------------------------------------------------------- FP8 cache

def _torch_e4m3_table():
    import torch
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()


def check_e4m3_decode_matches_torch(o):
    """Every one of the 256 codes decodes to torch's float8_e4m3fn value (NaN at 0x7F, 0xFF)."""
    ref = _torch_e4m3_table()
    got = o.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def check_e4m3_encode_matches_torch(o):
    """Encoding agrees with torch's conversion over magnitudes from the
    subnormals to 448; exact midpoints go to the even code; magnitudes above
    448 saturate to +-448."""
    import torch
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(50000) * np.exp(rng.uniform(-13, 7, 50000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.e4m3_encode(x), ref)
    tab = _torch_e4m3_table()[:0x7F].astype(np.float64)  # non-negative finite values, increasing
    mid = ((tab[:-1] + tab[1:]) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (tab[:-1] + tab[1:]) / 2)  # midpoints exact in fp32
    codes = o.e4m3_encode(mid)
    lo = np.arange(0x7E, dtype=np.uint8)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)  # the neighbour with an even mantissa
    assert np.array_equal(codes, expect)
    assert np.array_equal(o.e4m3_encode(-mid), expect | 0x80)
    big = np.array([448.0, 449.0, 463.9, 1e4, 3e38], dtype=np.float32)
    assert np.array_equal(o.e4m3_encode(big), np.full(5, 0x7E, np.uint8))
    assert np.array_equal(o.e4m3_encode(-big), np.full(5, 0xFE, np.uint8))


V_ORDER = [0, 1, 8, 9, 2, 3, 10, 11, 4, 5, 12, 13, 6, 7, 14, 15]  # token slot at each value byte


def fp8_tile_views(tiles):
    """Key codes [nb][Hkv][16][128], value codes [nb][Hkv][128][16] (natural slot
    order), key and value scales [nb][Hkv][16] read out of FP8 tiles, following
    the layout as the header defines it."""
    s = np.arange(16)[:, None]
    d = np.arange(128)[None, :]
    kb = 128 * s + 16 * ((d // 16) ^ (s % 8)) + d % 16               # [16][128]
    vpos = np.array([V_ORDER.index(x) for x in range(16)])
    vb = 2048 + 16 * d.T + vpos[None, :]                               # [128][16]
    k = tiles[:, :, kb]
    v = tiles[:, :, vb]
    ks = np.ascontiguousarray(tiles[:, :, 4096:4160]).view(np.float32)
    vs = np.ascontiguousarray(tiles[:, :, 4160:4224]).view(np.float32)
    return k, v, ks, vs


def fp8_case(seed, B, Hkv, ctx_lens, permute=True):
    """Random FP8 tiles for every slot (no NaN codes) and the table."""
    rng = np.random.default_rng(seed)
    L = np.asarray(ctx_lens, dtype=np.int32)
    max_blocks = int(-(-L.max() // wl.BLOCK))
    num_blocks, table = wl.layout_blocks(L, max_blocks, spare=2, permute=permute, rng=rng)
    codes = np.concatenate([np.arange(0x7F), np.arange(0x80, 0xFF)]).astype(np.uint8)
    tiles = rng.choice(codes, size=(num_blocks, Hkv, 4224)).astype(np.uint8)
    sc = rng.uniform(1e-3, 2e-2, (num_blocks, Hkv, 32)).astype(np.float32)
    tiles[:, :, 4096:] = sc.view(np.uint8).reshape(num_blocks, Hkv, 128)
    return dict(tiles=tiles, block_table=table, ctx_lens=L, rng=rng)


def check_kv_append_fp8_quantization(o):
    """Each appended row: scale = max|x| / 448 in fp32, codes = torch's E4M3 of
    x / scale, keys and values at the row's slot of the tile layout; the largest
    entry maps to +-448; every other byte of the tiles is untouched."""
    import torch
    B, Hkv, D, q_len = 3, 2, 128, 2
    c = fp8_case(21, B, Hkv, [5, 17, 32])
    before = (c["ctx_lens"] - q_len).astype(np.int32)
    rng = c["rng"]
    k_new = wl.f32_to_bf16(rng.standard_normal((B, q_len, Hkv, D), dtype=np.float32))
    v_new = wl.f32_to_bf16(3 * rng.standard_normal((B, q_len, Hkv, D), dtype=np.float32))
    v_new[0, 0, 0] = 0  # an all-zero row: scale 0, codes 0
    out = o.kv_append_fp8(c["tiles"], c["block_table"], before, k_new, v_new)
    kc, vc, ks, vs = fp8_tile_views(out)
    kc0, vc0, ks0, vs0 = fp8_tile_views(c["tiles"])
    touched = np.zeros(ks.shape, dtype=bool)
    for b in range(B):
        for j in range(q_len):
            s = before[b] + j
            blk, slot = c["block_table"][b, s // wl.BLOCK], s % wl.BLOCK
            for g in range(Hkv):
                touched[blk, g, slot] = True
                for x_bits, codes, scale in ((k_new[b, j, g], kc[blk, g, slot, :], ks[blk, g, slot]),
                                             (v_new[b, j, g], vc[blk, g, :, slot], vs[blk, g, slot])):
                    x = wl.bf16_to_f32(x_bits)
                    amax = np.float32(np.abs(x).max())
                    assert scale == np.float32(amax / np.float32(448.0))
                    if amax == 0:
                        assert not codes.any()
                        continue
                    ref = torch.from_numpy((x / scale).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
                    assert np.array_equal(codes, ref.numpy())
                    assert (codes[np.argmax(np.abs(x))] & 0x7F) == 0x7E
                    deq = o.e4m3_decode(codes).astype(np.float64) * scale
                    normal = np.abs(x) >= scale * 2.0 ** -6
                    assert np.all(np.abs(deq - x)[normal] <= 2.0 ** -4 * np.abs(x)[normal])
                    assert np.all(np.abs(deq - x)[~normal] <= 2.0 ** -10 * scale)
    assert np.array_equal(ks[~touched], ks0[~touched]) and np.array_equal(vs[~touched], vs0[~touched])
    assert np.array_equal(kc[~touched], kc0[~touched])
    assert np.array_equal(vc.transpose(0, 1, 3, 2)[~touched], vc0.transpose(0, 1, 3, 2)[~touched])
    # the views cover every byte of a tile exactly once
    idx = np.arange(4224, dtype=np.int64)[None, None, :]
    kb, vb, ksb, vsb = fp8_tile_views(np.broadcast_to(idx, (1, 1, 4224)).astype(np.int64))[:2] + (None, None)
    covered = np.concatenate([kb.ravel(), vb.ravel(), np.arange(4096, 4224)])
    assert np.array_equal(np.sort(covered), np.arange(4224))


def check_attn_fp8_matches_sdpa(o):
    """Attention over an FP8 cache equals torch's scaled_dot_product_attention
    (float64) on the cache dequantised with torch's E4M3 table."""
    import torch
    import torch.nn.functional as F
    tab = torch.from_numpy(_torch_e4m3_table().astype(np.float64))
    for (Hq, Hkv, q_len, causal, L, seed) in [(4, 2, 1, False, [17, 1, 40], 31), (8, 2, 5, True, [5, 33, 20], 32)]:
        D = 128
        c = fp8_case(seed, len(L), Hkv, L)
        kc, vc, ks, vs = fp8_tile_views(c["tiles"])
        q = wl.f32_to_bf16(c["rng"].standard_normal((len(L), q_len, Hq, D), dtype=np.float32))
        scale = 1.0 / math.sqrt(D)
        out = o.decode_attn_fp8(c["tiles"], c["block_table"], c["ctx_lens"], q, scale, causal)
        g = Hq // Hkv
        for b, Lb in enumerate(L):
            t = np.arange(Lb)
            blocks, slots = c["block_table"][b, t // wl.BLOCK], t % wl.BLOCK
            k = tab[torch.from_numpy(kc[blocks, :, slots, :].astype(np.int64))] * \
                torch.from_numpy(ks[blocks, :, slots].astype(np.float64))[..., None]
            v = tab[torch.from_numpy(vc[blocks, :, :, slots].astype(np.int64))] * \
                torch.from_numpy(vs[blocks, :, slots].astype(np.float64))[..., None]
            k = k.permute(1, 0, 2).repeat_interleave(g, dim=0)
            v = v.permute(1, 0, 2).repeat_interleave(g, dim=0)
            qq = torch.from_numpy(wl.bf16_to_f32(q[b]).astype(np.float64)).permute(1, 0, 2)
            mask = None
            if causal:
                mask = torch.arange(Lb)[None, :] < (Lb - q_len + torch.arange(q_len)[:, None] + 1)
            ref = F.scaled_dot_product_attention(qq, k, v, attn_mask=mask, scale=scale)
            err = (torch.from_numpy(out[b]).permute(1, 0, 2) - ref).abs().max().item()
            assert err < 1e-10, f"fp8 attention vs SDPA: {err}"


# --------------------------------------------------------------------- RoPE

def check_rope_identity_at_position_zero(o):
    """Position 0 rotates by angle 0 in every pair: the rows come back unchanged."""
    x = np.random.default_rng(41).standard_normal((4, 128)).astype(np.float32)
    assert np.array_equal(o.rope(x, np.zeros(4, np.int32)), x)
    xb = wl.f32_to_bf16(x)
    assert np.array_equal(o.rope(xb, np.zeros(4, np.int32)), wl.bf16_to_f32(xb))


def check_rope_matches_complex_rotation(o):
    """Rotate-half RoPE equals multiplying z_i = x_i + i x_(i+D/2) by
    exp(i pos base^(-2i/D)) (numpy complex arithmetic, float64)."""
    rng = np.random.default_rng(42)
    for D, base in ((128, 10000.0), (64, 500000.0)):
        x = rng.standard_normal((6, D)).astype(np.float32)
        pos = np.array([0, 1, 7, 100, 2047, 4095], np.int32)
        h = D // 2
        z = x[:, :h].astype(np.float64) + 1j * x[:, h:].astype(np.float64)
        theta = base ** (-2.0 * np.arange(h) / D)
        zr = z * np.exp(1j * pos[:, None] * theta[None, :])
        ref = np.concatenate([zr.real, zr.imag], axis=1)
        got = o.rope(x, pos, base).astype(np.float64)
        assert np.abs(got - ref).max() <= 4e-7 * max(1.0, np.abs(ref).max())


def check_rope_relative_position(o):
    """<rope(q, m), rope(k, n)> depends only on m - n: it equals <rope(q, m - n), k>."""
    rng = np.random.default_rng(43)
    q = rng.standard_normal((5, 128)).astype(np.float32)
    k = rng.standard_normal((5, 128)).astype(np.float32)
    m = np.array([10, 300, 4000, 17, 2], np.int32)
    n = np.array([3, 299, 1, 17, 0], np.int32)
    lhs = np.einsum("rd,rd->r", o.rope(q, m).astype(np.float64), o.rope(k, n).astype(np.float64))
    rhs = np.einsum("rd,rd->r", o.rope(q, m - n).astype(np.float64), k.astype(np.float64))
    assert np.abs(lhs - rhs).max() < 1e-4, np.abs(lhs - rhs).max()


def check_rope_pairs_keep_their_norm(o):
    """Each (i, i + D/2) pair is rotated, not scaled."""
    rng = np.random.default_rng(44)
    x = rng.standard_normal((3, 128)).astype(np.float32)
    r = o.rope(x, np.array([5, 999, 3000], np.int32)).astype(np.float64)
    n0 = np.hypot(x[:, :64].astype(np.float64), x[:, 64:].astype(np.float64))
    n1 = np.hypot(r[:, :64], r[:, 64:])
    assert np.abs(n1 - n0).max() < 1e-5


def check_fp8_append_from_float_rows(o):
    """FP8 rows given in float32 quantise the same way as bf16 rows holding the
    same values."""
    c = fp8_case(45, 2, 2, [3, 20])
    rng = c["rng"]
    kb = wl.f32_to_bf16(rng.standard_normal((2, 1, 2, 128), dtype=np.float32))
    vb = wl.f32_to_bf16(rng.standard_normal((2, 1, 2, 128), dtype=np.float32))
    before = (c["ctx_lens"] - 1).astype(np.int32)
    a = o.kv_append_fp8(c["tiles"], c["block_table"], before, kb, vb)
    b = o.kv_append_fp8(c["tiles"], c["block_table"], before, wl.bf16_to_f32(kb), wl.bf16_to_f32(vb))
    assert np.array_equal(a, b)


# ------------------------------------------------------------- audio head

def _mish_identity(x):
    """Mish through tanh(ln n) = (n^2 - 1) / (n^2 + 1) with n = 1 + e^x."""
    x = np.asarray(x, dtype=np.float64)
    n2 = (1.0 + np.exp(np.minimum(x, 300.0))) ** 2
    return x * (n2 - 1.0) / (n2 + 1.0)


def check_mish_closed_forms(o):
    """Mish against the algebraic form of tanh(softplus), its published minimum
    (about -0.30884 at x = -1.1924), slope 0.6 at zero (tanh(ln 2)), and its
    limits (x for large x, x e^x for very negative x)."""
    x = np.linspace(-20.0, 20.0, 4001)
    m = o.mish(x)
    ref = _mish_identity(x)
    assert np.all(np.abs(m - ref) <= 1e-13 * np.maximum(1.0, np.abs(ref)))
    assert o.mish([0.0])[0] == 0.0
    i = int(np.argmin(m))
    assert abs(x[i] - (-1.1924)) < 0.011 and abs(m[i] - (-0.30884)) < 1e-4
    eps = 1e-7
    slope = (o.mish([eps])[0] - o.mish([-eps])[0]) / (2 * eps)
    assert abs(slope - 0.6) < 1e-8
    assert o.mish([50.0])[0] == 50.0
    big = o.mish([-40.0])[0]
    assert abs(big / (-40.0 * math.exp(-40.0)) - 1.0) < 1e-12


def check_bf16_round_matches_torch(o):
    """Rounding to bfloat16 equals torch's conversion for float32-exact inputs
    (one rounding either way), ties to the even significand, specials kept."""
    import torch
    rng = np.random.default_rng(61)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-6, 6, 20000),
                        # exact midpoints between neighbouring bfloat16 values
                        (np.arange(1, 2000) * 2 + 1).astype(np.float64) * 2.0 ** -9,
                        -(np.arange(1, 2000) * 2 + 1).astype(np.float64) * 2.0 ** -9,
                        [0.0, -0.0, 1e-40, -3e-39, 3.3e38]]).astype(np.float32)
    got = o.bf16_round(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    assert o.bf16_round([1.0 + 2.0 ** -8])[0] == 0x3F80      # tie -> even (1.0)
    assert o.bf16_round([1.0 + 3 * 2.0 ** -8])[0] == 0x3F82  # tie -> even (1.015625)
    assert o.bf16_round([math.inf])[0] == 0x7F80 and o.bf16_round([-math.inf])[0] == 0xFF80


def check_audio_expand_matches_matmul(o):
    """z = bf16(Mish(h W1^T + b1)) against a numpy float64 matmul, the algebraic
    Mish and a nearest-value test of the rounding; the bias shifts the input."""
    rng = np.random.default_rng(62)
    R, H, F = 3, 64, 40
    h = wl.f32_to_bf16(rng.standard_normal((R, H), dtype=np.float32))
    W1 = wl.f32_to_bf16((rng.standard_normal((F, H)) / 8).astype(np.float32))
    b1 = rng.standard_normal(F).astype(np.float32)
    pre = wl.bf16_to_f32(h).astype(np.float64) @ wl.bf16_to_f32(W1).astype(np.float64).T + b1
    z, m = o.audio_expand(h, W1, b1)
    assert np.all(np.abs(m - _mish_identity(pre)) <= 1e-12 * np.maximum(1.0, np.abs(m)))
    zf = wl.bf16_to_f32(z).astype(np.float64)
    # every z is a nearest bfloat16 of m: no neighbour one step away is closer
    bits = z.astype(np.int64)
    for step in (-1, 1):
        nb = wl.bf16_to_f32((bits + step).astype(np.uint16)).astype(np.float64)
        assert np.all(np.abs(zf - m) <= np.abs(nb - m))
    z0, m0 = o.audio_expand(h, W1, None)
    assert np.allclose(m0, _mish_identity(pre - b1), rtol=1e-12, atol=1e-12)
    z1, _ = o.audio_expand(h, W1, np.zeros(F, np.float32))
    assert np.array_equal(z0, z1)


def _masked_reference(h, W, b, n_tail, tail_allowed):
    """numpy: float32 logits, masked tail ids removed, lowest index on ties."""
    lg = (wl.bf16_to_f32(h).astype(np.float64) @ wl.bf16_to_f32(W).astype(np.float64).T
          + (0.0 if b is None else b.astype(np.float64))).astype(np.float32)
    V = W.shape[0]
    keep = np.ones(lg.shape, bool)
    if tail_allowed is not None:
        for j in range(n_tail):
            keep[:, V - n_tail + j] = (tail_allowed >> j) & 1 == 1
    masked = np.where(keep, lg.astype(np.float64), -np.inf)
    return lg, masked, np.argmax(masked, axis=1)


def check_head_masked_bias_and_tail(o):
    """Biased, masked selection against numpy's argmax over the allowed ids;
    a tail id with a dominant bias wins exactly when its mask bit is set, and
    mask bit j governs id V - n_tail + j."""
    rng = np.random.default_rng(63)
    R, H, V, n_tail = 6, 32, 50, 3
    h = wl.f32_to_bf16(rng.standard_normal((R, H), dtype=np.float32))
    W = wl.f32_to_bf16((rng.standard_normal((V, H)) / 4).astype(np.float32))
    b = (rng.standard_normal(V) / 10).astype(np.float32)
    ta = rng.integers(0, 8, R).astype(np.uint32)
    res = o.head_select_masked(h, W, b, n_tail=n_tail, tail_allowed=ta, want_logits=True)
    lg, masked, ref_ids = _masked_reference(h, W, b, n_tail, ta)
    assert np.array_equal(res["logits"], lg)
    assert np.array_equal(res["ids"], ref_ids)
    # dominant tail biases: row r picks the highest allowed tail id bit
    b2 = b.copy()
    b2[V - n_tail:] = [100.0, 200.0, 300.0]
    ta2 = np.array([0, 1, 2, 4, 3, 7], np.uint32)
    res2 = o.head_select_masked(h, W, b2, n_tail=n_tail, tail_allowed=ta2)
    expect = []
    for r, m in enumerate(ta2):
        allowed = [j for j in range(n_tail) if (m >> j) & 1]
        # no tail id allowed: the codebook's own argmax (its biases are unchanged)
        expect.append(V - n_tail + max(allowed) if allowed else int(np.argmax(lg[r, :V - n_tail])))
    assert list(res2["ids"]) == expect
    # no mask and no bias: plain selection over the matmul
    res3 = o.head_select_masked(h, W)
    assert np.array_equal(res3["ids"], np.argmax(_masked_reference(h, W, None, 0, None)[0], axis=1))


def check_head_masked_gumbel(o):
    """Gumbel selection with a mask draws from softmax(logits / T) restricted to
    the allowed ids: the keys are the oracle's noise added to logits / T, and
    the frequencies pass a chi-square test with masked ids never drawn."""
    rng = np.random.default_rng(64)
    H, V, n_tail, T = 16, 12, 2, 0.8
    W = wl.f32_to_bf16((rng.standard_normal((V, H)) / 2).astype(np.float32))
    h1 = wl.f32_to_bf16(rng.standard_normal((1, H), dtype=np.float32))
    rows = 3000
    h = np.repeat(h1, rows, axis=0)
    ta = np.full(rows, 0b10, np.uint32)   # id V-2 masked, id V-1 allowed
    seeds = np.arange(rows, dtype=np.uint64) + 7
    res = o.head_select_masked(h, W, None, "gumbel", T, seeds, np.zeros(rows, np.uint64), n_tail, ta,
                               want_logits=True)
    lg = res["logits"][0].astype(np.float64)
    assert not np.any(res["ids"] == V - 2)
    p = _softmax64(np.where(np.arange(V) == V - 2, -np.inf, lg), T)
    counts = np.bincount(res["ids"], minlength=V)
    keep = p > 0
    assert _chi2_p(counts[keep], p[keep]) > 1e-3
    # row 0's key is its logit / T plus the oracle's Gumbel noise for that id
    v = int(res["ids"][0])
    key = np.float32(np.float32(res["logits"][0, v]) / np.float32(T)) + np.float32(o.gumbel(int(seeds[0]), 0, 0, 0, v))
    assert res["best"][0] == np.float32(key)


def check_audio_head_composition(o):
    """The two-layer head selects over z W2^T + b2 with z from the first layer."""
    rng = np.random.default_rng(65)
    R, H, F, V = 4, 32, 24, 20
    h = wl.f32_to_bf16(rng.standard_normal((R, H), dtype=np.float32))
    W1 = wl.f32_to_bf16((rng.standard_normal((F, H)) / 6).astype(np.float32))
    W2 = wl.f32_to_bf16((rng.standard_normal((V, F)) / 5).astype(np.float32))
    b1 = rng.standard_normal(F).astype(np.float32)
    b2 = rng.standard_normal(V).astype(np.float32)
    out = o.audio_head(h, W1, b1, W2, b2, n_tail=2, tail_allowed=np.array([0, 1, 2, 3], np.uint32))
    z, _ = o.audio_expand(h, W1, b1)
    assert np.array_equal(out["z"], z)
    _, _, ref = _masked_reference(z, W2, b2, 2, np.array([0, 1, 2, 3], np.uint32))
    assert np.array_equal(out["ids"], ref)


# --------------------------------------------------------- code predictor

def predictor_case(seed, R=3, H=64, Hq=4, Hkv=2, D=16, V=40, n_steps=15):
    rng = np.random.default_rng(seed)
    F = (Hq + 2 * Hkv) * D
    return dict(
        x0=wl.f32_to_bf16(rng.standard_normal((R, H), dtype=np.float32)),
        Wqkv=wl.f32_to_bf16((rng.standard_normal((F, H)) / 6).astype(np.float32)),
        W=wl.f32_to_bf16((rng.standard_normal((n_steps, V, Hq * D)) / 4).astype(np.float32)),
        E=wl.f32_to_bf16(rng.standard_normal((n_steps, V, H)).astype(np.float32)),
        Hq=Hq, Hkv=Hkv, D=D)


def check_code_predictor_stages(o):
    """Each step of the loop against library routines: the projection is a
    numpy float64 matmul rounded to bf16, the attention torch's float64 SDPA
    (GQA, keys and values of steps 0..i) rounded to bf16, the token numpy's
    argmax of float32 logits, and the next input the chosen token's row of
    that step's embedding; step 0 attends to one token, so o equals its v."""
    import torch
    c = predictor_case(71)
    Hq, Hkv, D = c["Hq"], c["Hkv"], c["D"]
    res = o.code_predictor(c["x0"], c["Wqkv"], c["W"], c["E"], Hq, Hkv, want_trace=True)
    n_steps, R = res["tokens"].shape
    HO, F = Hq * D, (Hq + 2 * Hkv) * D
    f64 = lambda b: wl.bf16_to_f32(b).astype(np.float64)
    Wqkv, W, E = f64(c["Wqkv"]), f64(c["W"]), f64(c["E"])
    for r in range(R):
        x = f64(c["x0"][r])
        ks, vs = [], []
        for i in range(n_steps):
            tr = res["trace"][i, r]
            qkv = f64(o.bf16_round(Wqkv @ x))
            assert np.array_equal(tr[:F], qkv)
            q = qkv[:HO].reshape(Hq, D)
            ks.append(qkv[HO:HO + Hkv * D].reshape(Hkv, D))
            vs.append(qkv[HO + Hkv * D:].reshape(Hkv, D))
            K = torch.from_numpy(np.repeat(np.stack(ks, 1), Hq // Hkv, axis=0))   # [Hq][t][D]
            Vv = torch.from_numpy(np.repeat(np.stack(vs, 1), Hq // Hkv, axis=0))
            att = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q)[:, None, :], K, Vv, scale=1.0 / math.sqrt(D))[:, 0, :].numpy()
            ob = o.bf16_round(att.reshape(-1))
            assert np.array_equal(tr[F:], f64(ob))
            if i == 0:
                assert np.array_equal(tr[F:], np.repeat(vs[0], Hq // Hkv, axis=0).reshape(-1))
            logits = (W[i] @ tr[F:]).astype(np.float32)
            assert res["tokens"][i, r] == int(np.argmax(logits))
            x = E[i, res["tokens"][i, r]]


def check_code_predictor_gumbel_keys(o):
    """Gumbel mode: step i's token maximises float32(logit) / T plus the noise
    of counter position i + 1, and best holds that key."""
    c = predictor_case(72, R=2, V=24, n_steps=6)
    T = 0.8
    seed = np.array([11, 12], np.uint64)
    step = np.array([5, 9], np.uint64)
    res = o.code_predictor(c["x0"], c["Wqkv"], c["W"], c["E"], c["Hq"], c["Hkv"], "gumbel", T, seed, step,
                           want_trace=True)
    F = (c["Hq"] + 2 * c["Hkv"]) * c["D"]
    W = wl.bf16_to_f32(c["W"]).astype(np.float64)
    for i in range(6):
        for r in range(2):
            logits = (W[i] @ res["trace"][i, r, F:]).astype(np.float32)
            keys = np.array([np.float32(logits[v] / np.float32(T)) +
                             np.float32(o.gumbel(int(seed[r]), int(step[r]), 0, i + 1, v)) for v in range(24)],
                            np.float32)
            assert res["tokens"][i, r] == int(np.argmax(keys))
            assert res["best"][i, r] == keys.max()


def check_code_predictor_uniform_attention(o):
    """Zero key projections make every score zero: o is the bf16 mean of the
    values of steps 0..i (per KV head)."""
    c = predictor_case(73, R=2, n_steps=8)
    Hq, Hkv, D = c["Hq"], c["Hkv"], c["D"]
    HO = Hq * D
    Wqkv = c["Wqkv"].copy()
    Wqkv[HO:HO + Hkv * D] = 0
    res = o.code_predictor(c["x0"], Wqkv, c["W"], c["E"], Hq, Hkv, want_trace=True)
    F = (Hq + 2 * Hkv) * D
    for r in range(2):
        vs = []
        for i in range(8):
            tr = res["trace"][i, r]
            assert not tr[HO:HO + Hkv * D].any()
            vs.append(tr[HO + Hkv * D:F].reshape(Hkv, D))
            mean = np.repeat(np.mean(np.stack(vs), axis=0), Hq // Hkv, axis=0).reshape(-1)
            # a nearest bf16 of the mean (the mean of bf16 values can sit on a
            # rounding midpoint, where the summation order picks the side)
            got = tr[F:]
            half_ulp = np.abs(wl.bf16_to_f32(o.bf16_round(mean)).astype(np.float64)) * 2.0 ** -8
            assert np.all(np.abs(got - mean) <= half_ulp * (1 + 1e-9) + 1e-300)


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
