"""Captured steps for a set of batch sizes (tts_step_graph_set) against the oracle.

Streams beyond the active ones of a launch are padded onto a scratch block;
cohorts larger than the largest captured size run one after another.  Ids of
the active streams must match the oracle's step (append, attention, head)
except at near-ties, and the pool must hold exactly the oracle's appended
rows outside the scratch block.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import compare_ids, dev, host

pytestmark = pytest.mark.gpu


def _host_tensor(x: np.ndarray) -> torch.Tensor:
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    if x.dtype == np.uint64:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int64))
    return torch.from_numpy(np.ascontiguousarray(x))


def test_graph_set_sizes_padding_and_cohorts(orc):
    from decode_step_gb300 import binding as bd
    from decode_step_gb300.step import DecodeStep, GraphedStepSet
    n_all, B = 100, 64
    w = wl.custom(3, B=n_all, ctx_lo=30, ctx_hi=400, permute_table=True)
    inp = wl.make_inputs(w, seed=2024, with_verify=False)
    table = inp["block_table"]
    used = set(int(x) for x in table[table >= 0].ravel())
    scratch = min(set(range(inp["num_blocks"])) - used)
    kp, vp = dev(inp["k_pool"]), dev(inp["v_pool"])
    cache = bd.KVCache(kp, vp)
    step = DecodeStep(cache, dev(inp["W"]), w.Hq, B, w.ctx_hi)
    names = ("block_table", "ctx_before", "ctx_lens", "q", "k_new", "v_new")
    arrays = {k: _host_tensor(inp[k]) for k in names}
    first = {k: arrays[k][:B].cuda() for k in names}
    gs = GraphedStepSet(step, first, sizes=[4, 16, B], scratch_block=scratch)
    # three streams: the size-4 graph with one padded stream
    ids3 = gs.step_streams({k: v[:3] for k, v in arrays.items()}).numpy()
    # all hundred: a cohort of 64 and one of 36 (the size-64 graph, 28 padded)
    ids_all = gs.step_streams(arrays).numpy()
    assert int(step.err.item()) == 0
    rk, rv = orc.kv_append(inp["k_pool"], inp["v_pool"], table, inp["ctx_before"], inp["k_new"], inp["v_new"])
    attn = orc.decode_attn(rk, rv, table, inp["ctx_lens"], inp["q"], inp["scale"])
    h = wl.f32_to_bf16(attn.reshape(w.R, w.Hq * w.D).astype(np.float32))
    ref = orc.head_select(h, inp["W"], "argmax")
    hard, ties = compare_ids(ids_all, ref)
    print(f"[graph set] 100 streams: near-ties {ties}, hard mismatches {len(hard)}")
    assert not hard
    sub = {k: v[:3] for k, v in ref.items()}
    hard3, _ = compare_ids(ids3, sub)
    assert not hard3
    # every block but the scratch one holds exactly the oracle's pool
    keep = np.array([b != scratch for b in range(inp["num_blocks"])])
    gk, gv = host(kp), host(vp)
    assert np.array_equal(gk[keep].view(np.uint16), rk[keep].view(np.uint16))
    assert np.array_equal(gv[keep].view(np.uint16), rv[keep].view(np.uint16))


def test_graph_set_rejects_bad_sizes(orc):
    from decode_step_gb300 import binding as bd
    from decode_step_gb300.step import DecodeStep, GraphedStepSet
    w = wl.custom(3, B=8, ctx_lo=30, ctx_hi=100)
    inp = wl.make_inputs(w, seed=7, with_verify=False)
    cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
    step = DecodeStep(cache, dev(inp["W"]), w.Hq, 8, w.ctx_hi)
    first = {k: dev(inp[k]) for k in ("block_table", "ctx_before", "ctx_lens", "q", "k_new", "v_new")}
    with pytest.raises(ValueError):
        GraphedStepSet(step, first, sizes=[4, 6], scratch_block=0)      # largest is not B
    with pytest.raises(bd.TTSError):
        GraphedStepSet(step, first, sizes=[4, 4, 8], scratch_block=0)   # not strictly increasing
    gs = GraphedStepSet(step, first, sizes=[2, 8], scratch_block=0)
    with pytest.raises(ValueError):
        gs.launch(9)
