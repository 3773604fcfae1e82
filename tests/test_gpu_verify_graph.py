"""The captured step with its speculative verify stage.

A q_len = K + 1 causal step with a Gumbel head keeps the target logits of
every stream's K + 1 rows; the captured step then verifies the K drafts on
them.  Its accepted counts and next tokens (read from pinned host memory)
must equal the eager path's: tts_decode_step followed by tts_spec_verify on
the same inputs (the same kernels; the eager verify is checked against the
oracle elsewhere).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import dev, host

pytestmark = pytest.mark.gpu


def test_captured_verify_matches_eager():
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
    print(f"[captured verify] accepted {n1.cpu().tolist()} next {x1.cpu().tolist()}")


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
