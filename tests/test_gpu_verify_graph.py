"""The captured step with its speculative verify stage.

A q_len = K + 1 causal step with a Gumbel head keeps the target logits of
every stream's K + 1 rows; the captured step then verifies the K drafts on
them.  Its accepted counts and next tokens (read from pinned host memory)
must equal the eager path's: tts_decode_step followed by tts_spec_verify on
the same inputs.  Each stage of the captured step is also compared with the
oracle on the same inputs: its attention with the oracle's attention, its ids
and logits with the oracle's head over the step's own attention output, its
accepted counts and next tokens with the oracle's verify over the step's own
target logits.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import ATOL, NEAR_TIE, RTOL, as_f64, attn_errors, compare_ids, dev, host, rel_where_binding

pytestmark = pytest.mark.gpu


def test_captured_verify_matches_eager(orc, parity):
    from decode_step_gb300 import binding as bd
    from decode_step_gb300.step import DecodeStep, GraphedStep
    w = wl.custom(5, B=8, ctx_lo=40, ctx_hi=300, permute_table=True)
    inp = wl.make_inputs(w, seed=4242, with_verify=True)
    K, T = w.K, w.T

    def fresh():
        cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
        return DecodeStep(cache, dev(inp["W"]), w.Hq, w.B, w.ctx_hi, q_len=w.q_len, causal=True,
                          mode=bd.TTS_GUMBEL, temperature=T)

    names = ("block_table", "ctx_before", "ctx_lens", "q", "k_new", "v_new", "seed", "step",
             "draft_probs", "draft_tokens", "vseed", "vstep")
    d = {k: dev(inp[k]) for k in names}
    # eager
    s1 = fresh()
    logits = torch.empty((w.R, w.V), dtype=torch.float32, device="cuda")
    ids1 = s1(d["block_table"], d["ctx_before"], d["ctx_lens"], d["q"], d["k_new"], d["v_new"],
              seed=d["seed"], step=d["step"], logits_out=logits).clone()
    n1 = torch.empty(w.B, dtype=torch.int32, device="cuda")
    x1 = torch.empty(w.B, dtype=torch.int32, device="cuda")
    bd.tts_spec_verify(logits.view(w.B, w.q_len, w.V), d["draft_probs"], d["draft_tokens"], T, d["vseed"],
                       d["vstep"], n1, x1)
    torch.cuda.synchronize()
    # captured
    s2 = fresh()
    g = GraphedStep(s2, d, verify_temperature=T)
    ids2 = g().clone()
    assert torch.equal(ids2, ids1.cpu())
    assert torch.equal(g.n_accepted_host, n1.cpu())
    assert torch.equal(g.next_token_host, x1.cpu())
    assert torch.equal(g.logits, logits)
    # a second launch reproduces it
    g()
    assert torch.equal(g.n_accepted_host, n1.cpu()) and torch.equal(g.next_token_host, x1.cpu())
    assert int(s1.err.item()) == 0 and int(s2.err.item()) == 0

    # ---- the captured step against the oracle, stage by stage
    kp, vp = orc.kv_append(inp["k_pool"], inp["v_pool"], inp["block_table"], inp["ctx_before"],
                           inp["k_new"], inp["v_new"])
    ref_attn = orc.decode_attn(kp, vp, inp["block_table"], inp["ctx_lens"], inp["q"], 1.0 / math.sqrt(w.D),
                               True)
    got_attn = as_f64(host(s2.out), "bf16")
    bad, mx_abs, mx_rel = attn_errors(got_attn, ref_attn)
    parity("captured verify step attention", max_abs=mx_abs, max_rel=mx_rel)
    assert bad == 0 and mx_abs <= ATOL and rel_where_binding(got_attn, ref_attn) <= RTOL
    h = host(s2.out).reshape(w.R, -1)
    ref_head = orc.head_select(h, inp["W"], "gumbel", T, inp["seed"], inp["step"], want_logits=True)
    hard, ties = compare_ids(ids2.numpy(), ref_head)
    parity("captured verify step head", rows=w.R, near_ties=ties, hard=len(hard))
    assert not hard, f"captured head ids differ from the oracle at rows {hard}"
    assert np.allclose(host(g.logits), ref_head["logits"], rtol=1e-4, atol=1e-4)
    tl = host(g.logits).reshape(w.B, w.q_len, w.V)
    ref_v = orc.spec_verify(tl, inp["draft_probs"], inp["draft_tokens"], T, inp["vseed"], inp["vstep"])
    tie = (ref_v["gap_accept"] < NEAR_TIE) | (ref_v["gap_resid"] < NEAR_TIE)
    badv = (g.n_accepted_host.numpy() != ref_v["n_accepted"]) | (g.next_token_host.numpy() != ref_v["next_token"])
    parity("captured verify step verify", streams=w.B, near_ties=int(tie.sum()), hard=int((badv & ~tie).sum()))
    assert not (badv & ~tie).any(), f"captured verify differs from the oracle at {np.nonzero(badv & ~tie)[0]}"


def test_captured_verify_rejects_bad_arguments():
    from decode_step_gb300 import binding as bd
    from decode_step_gb300.step import DecodeStep, GraphedStep
    w = wl.custom(5, B=2, ctx_lo=40, ctx_hi=100)
    inp = wl.make_inputs(w, seed=9, with_verify=True)
    cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
    step = DecodeStep(cache, dev(inp["W"]), w.Hq, w.B, w.ctx_hi, q_len=w.q_len, causal=True,
                      mode=bd.TTS_GUMBEL, temperature=w.T)
    names = ("block_table", "ctx_before", "ctx_lens", "q", "k_new", "v_new", "seed", "step",
             "draft_probs", "draft_tokens", "vseed", "vstep")
    d = {k: dev(inp[k]) for k in names}
    with pytest.raises(bd.TTSError):
        GraphedStep(step, d, verify_temperature=0.0)   # the verify temperature must be positive
