"""tts_decode_attn_noalloc: decode attention for callers that cannot call
cudaMalloc where they run a step (an engine that has handed all free device
memory to its KV pool, a plugin host that gives the library no allocator, a
real-time loop that cannot absorb cudaMalloc's synchronisation).  It must give
the same output as tts_decode_attn with a caller workspace, call after call,
although every call reuses the one static scratch array.

Kept in a file of its own that pytest collects last, so a run that stops at
the first failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import Uploaded, as_f64, attn_errors, host

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from decode_step_gb300 import binding as bd


def _attn_with_workspace(u, cache, w):
    ws = torch.zeros(bd.tts_decode_attn_workspace_size(w.B, w.q_len, w.Hq, w.Hkv, w.D, w.ctx_hi),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(u.q)
    bd.tts_decode_attn(cache, u.table, u.ctx_lens, w.ctx_hi, u.q, out, ws, 1.0 / math.sqrt(w.D),
                       w.causal)
    return out


# The acoustic-b64 step and the causal 5-row speculative-verify step.
CASES = {"acoustic-b64": wl.WORKLOADS[3], "verify-b64": wl.WORKLOADS[5]}


def _check_noalloc_twice(name):
    inp = wl.make_inputs(CASES[name], with_head=False, with_verify=False)
    w = inp["workload"]
    u = Uploaded(inp)
    cache = bd.KVCache(u.k_pool, u.v_pool)
    bd.tts_kv_append(cache, u.table, u.ctx_before, u.k_new, u.v_new)
    ref = as_f64(host(_attn_with_workspace(u, cache, w)), w.dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):  # the second call sees the scratch as the first left it
        out = torch.full_like(u.q, float("nan"))
        bd.tts_decode_attn_noalloc(cache, u.table, u.ctx_lens, w.ctx_hi, u.q, out,
                                   1.0 / math.sqrt(w.D), w.causal, err=err)
        torch.cuda.synchronize()
        got = as_f64(host(out), w.dtype)
        assert np.isfinite(got).all(), f"{name} call {call}: non-finite output"
        bad, mx_abs, _ = attn_errors(got, ref)
        assert bad == 0, f"{name} call {call}: {bad} elements differ (max abs {mx_abs})"
    assert int(err.item()) == 0


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_workspace_entry_point(name):
    _check_noalloc_twice(name)


def test_noalloc_clears_tickets_left_by_a_larger_call():
    # verify-b64's 10-row partial slots reach ~19 MB into the array, across
    # the offset where acoustic-b64's split tickets sit (~3.8 MB), and leave
    # nonzero floats there.  The acoustic call must still start from zeroed
    # tickets and match the workspace entry point.
    _check_noalloc_twice("verify-b64")
    _check_noalloc_twice("acoustic-b64")


def test_noalloc_rejects_requests_beyond_the_static_scratch():
    # 16 query heads on one KV head: 16-row partials, about 20 MB > 16 MiB.
    w = wl.custom(4, B=256, Hq=16, Hkv=1, ctx_hi=4096)
    need = bd.tts_decode_attn_workspace_size(w.B, 1, w.Hq, w.Hkv, w.D, w.ctx_hi)
    assert need > 16 << 20
    pool = torch.zeros((4, w.Hkv, 16, w.D), dtype=torch.bfloat16, device="cuda")
    cache = bd.KVCache(pool, pool.clone())
    table = torch.zeros((w.B, 256), dtype=torch.int32, device="cuda")
    lens = torch.ones(w.B, dtype=torch.int32, device="cuda")
    q = torch.zeros((w.B, 1, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bd.TTSError) as e:
        bd.tts_decode_attn_noalloc(cache, table, lens, w.ctx_hi, q, torch.empty_like(q), 0.088)
    assert e.value.code == -6
