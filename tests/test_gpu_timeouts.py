"""The bounded on-device waits give up, flag TTS_ERRBIT_TIMEOUT and return.

A test-only stall (tts_test_set_stall) makes one wait wait for something that
never comes: 16 bytes more on an attention warp's first ring stage than its
copies deliver, or one arrival more at the code predictor's first grid
barrier than the grid has.  With a short wait limit the kernel must finish,
flag the timeout, and leave the context usable: the same call without the
stall then matches the oracle.  Nothing here faults, traps or hangs: every
wait is bounded and the stall only withholds a completion.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import ATOL, Uploaded, as_f64, attn_errors, dev, host

pytestmark = pytest.mark.gpu

LIMIT = 200_000  # SM clock cycles per wait, about 0.1 ms


@pytest.fixture
def bd():
    from decode_step_gb300 import binding
    yield binding
    binding.tts_test_set_stall(binding._lib.TEST_STALL_NONE)


def test_attention_ring_wait_times_out(orc, bd):
    w = wl.custom(3, B=8, ctx_lo=20, ctx_hi=400)
    inp = wl.make_inputs(w, seed=31, with_head=False, with_verify=False)
    u = Uploaded(inp)
    cache = bd.KVCache(u.k_pool, u.v_pool)
    bd.tts_kv_append(cache, u.table, u.ctx_before, u.k_new, u.v_new)
    ws = torch.zeros(bd.tts_decode_attn_workspace_size(w.B, w.q_len, w.Hq, w.Hkv, w.D, w.ctx_hi),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(u.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_test_set_stall(bd._lib.TEST_STALL_ATTN_RING, LIMIT)
    bd.tts_decode_attn(cache, u.table, u.ctx_lens, w.ctx_hi, u.q, out, ws, 1.0 / math.sqrt(w.D), False, err=err)
    torch.cuda.synchronize()           # the kernel returned
    assert int(err.item()) & bd._lib.ERRBIT_TIMEOUT
    # no stall: the context still works and the result is right
    bd.tts_test_set_stall(bd._lib.TEST_STALL_NONE)
    err.zero_()
    ws.zero_()                          # the stalled call may have left split tickets behind
    bd.tts_decode_attn(cache, u.table, u.ctx_lens, w.ctx_hi, u.q, out, ws, 1.0 / math.sqrt(w.D), False, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kp, vp = orc.kv_append(inp["k_pool"], inp["v_pool"], inp["block_table"], inp["ctx_before"], inp["k_new"],
                           inp["v_new"])
    ref = orc.decode_attn(kp, vp, inp["block_table"], inp["ctx_lens"], inp["q"], 1.0 / math.sqrt(w.D))
    bad, mx_abs, _ = attn_errors(as_f64(host(out), "bf16"), ref)
    assert bad == 0 and mx_abs <= ATOL


def test_predictor_grid_barrier_times_out(orc, bd):
    R, Hq, Hkv, V, n = 5, 2, 1, 112, 15
    H = Hq * 128
    inp = wl.code_predictor_inputs(R, H, Hq, Hkv, 128, V, n, seed=6100)
    args = [dev(inp[k]) for k in ("x0", "Wqkv", "W", "E")]
    tok = torch.full((n, R), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.tts_test_set_stall(bd._lib.TEST_STALL_PREDICTOR_GRID, LIMIT)
    bd.CodePredictor(*args, Hq, Hkv, tok, err=err).run()
    torch.cuda.synchronize()
    assert int(err.item()) & bd._lib.ERRBIT_TIMEOUT
    bd.tts_test_set_stall(bd._lib.TEST_STALL_NONE)
    err.zero_()
    bd.CodePredictor(*args, Hq, Hkv, tok, err=err).run()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = orc.code_predictor(inp["x0"], inp["Wqkv"], inp["W"], inp["E"], Hq, Hkv)
    got = host(tok)
    for r in range(R):          # up to each stream's first near-tie, as the predictor tests compare
        for i in range(n):
            if got[i, r] != ref["tokens"][i, r]:
                assert ref["best"][i, r] - ref["second"][i, r] < 1e-3
                break
