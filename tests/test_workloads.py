"""The seeded input generator: shapes, determinism, poisoning (CPU only)."""
import numpy as np

import workloads as wl


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-9, -2.5, np.inf, 0.0], dtype=np.float32)
    b = wl.f32_to_bf16(x)
    assert list(wl.bf16_to_f32(b)) == [1.0, 1.0, 1.0 + 2**-7, -2.5, np.inf, 0.0]
    assert np.isnan(wl.bf16_to_f32(wl.f32_to_bf16(np.array([np.nan], np.float32))))[0]


def test_tiny_workload_is_deterministic_and_shaped():
    a = wl.make_inputs(1)
    b = wl.make_inputs(1)
    w = wl.WORKLOADS[1]
    for k in ("q", "k_new", "v_new", "k_pool", "v_pool", "h", "W", "block_table", "ctx_lens"):
        assert np.array_equal(a[k], b[k], equal_nan=True), k
    assert a["q"].shape == (w.B, 1, w.Hq, w.D) and a["q"].dtype == np.float32
    assert a["W"].shape == (w.V, w.H)
    L = a["ctx_lens"]
    assert ((L >= 16) & (L <= 64)).all()
    assert np.array_equal(a["ctx_before"], L - 1)


def test_pool_poisoning_marks_exactly_the_empty_slots():
    w = wl.custom(3, B=6, ctx_lo=1, ctx_hi=70, q_len=2)
    inp = wl.make_inputs(w, seed=3, with_head=False)
    kp, table = inp["k_pool"], inp["block_table"]
    filled = ~np.isnan(wl.bf16_to_f32(kp[:, 0, :, 0]))
    expect = np.zeros_like(filled)
    for b, n in enumerate(inp["ctx_before"]):
        for s in range(int(n)):
            expect[table[b, s // 16], s % 16] = True
    assert np.array_equal(filled, expect)
    used = table[table >= 0]
    assert len(np.unique(used)) == len(used)


def test_verify_inputs():
    w = wl.custom(5, B=8, V=97, H=64)
    inp = wl.make_inputs(w, seed=1)
    assert inp["target_logits"].shape == (8, 5, 97)
    dp = inp["draft_probs"]
    assert dp.shape == (8, 4, 97) and np.allclose(dp.sum(-1), 1.0, atol=1e-5)
    assert ((inp["draft_tokens"] >= 0) & (inp["draft_tokens"] < 97)).all()
