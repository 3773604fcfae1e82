"""Two-layer audio head (tts_audio_head_select) on the GPU against the oracle.

The first layer's output z is bf16: the kernel sums in fp32 on the tensor
cores and applies Mish in fp32, the oracle sums and applies Mish in double and
rounds once, so a z element may differ only where the oracle's Mish value lies
within the fp32 summation error of a rounding midpoint.  Logits then differ by
at most a few of those flips; ids must match except at the oracle's near-ties.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import compare_ids, dev, host

pytestmark = pytest.mark.gpu

ERR_INVALID, ERR_UNSUPPORTED = -1, -2   # status codes of the C interface


@pytest.fixture(scope="module")
def bd():
    from decode_step_gb300 import binding
    return binding


def _run(bd, inp, R, F, V, n_tail, mode="argmax", T=0.0, logits=False, masked=True):
    z = torch.empty((R, F), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(R, dtype=torch.int32, device="cuda")
    best = torch.empty(R, dtype=torch.float32, device="cuda")
    lo = torch.empty((R, V), dtype=torch.float32, device="cuda") if logits else None
    ws = torch.zeros(bd.tts_head_workspace_size(R, V), dtype=torch.uint8, device="cuda")
    ta = dev(inp["tail_allowed"].view(np.int32)) if masked else None
    m = bd.TTS_GUMBEL if mode == "gumbel" else bd.TTS_ARGMAX
    for _ in range(2):  # twice: the workspace is left ready for the next call
        bd.tts_audio_head_select(dev(inp["h"]), dev(inp["W1"]), dev(inp["b1"]), dev(inp["W2"]), dev(inp["b2"]), z,
                                 ids, ws, mode=m, temperature=T, seed=dev(inp["seed"]), step=dev(inp["step"]),
                                 n_tail=n_tail, tail_allowed=ta, best=best, logits_out=lo)
        torch.cuda.synchronize()
    return host(z), host(ids), host(best), None if lo is None else host(lo)


def check_z(orc, inp, z_gpu, z_ref, mish_ref):
    """z equals the oracle's rounding except where the oracle's Mish value lies
    within the kernel's fp32 error of a rounding boundary: each differing
    element must be the rounding of some value within that error of the
    oracle's (between the roundings of m - tol and m + tol)."""
    bad = np.nonzero(z_gpu != z_ref)
    n = len(bad[0])
    if n:
        hf = np.abs(wl.bf16_to_f32(inp["h"]).astype(np.float64))
        wf = np.abs(wl.bf16_to_f32(inp["W1"]).astype(np.float64))
        mag = hf @ wf.T + np.abs(inp["b1"].astype(np.float64))     # sum |h_k w_k| + |b|
        g = wl.bf16_to_f32(z_gpu[bad]).astype(np.float64)
        m = mish_ref[bad]
        # fp32 sum error (a few 2^-24 per term, generously 2^-17 of the magnitude),
        # Mish's slope below 1.1, and its fp32 evaluation
        tol = 1.1 * 2.0 ** -17 * mag[bad] + 2.0 ** -20 * np.abs(m)
        lo = wl.bf16_to_f32(orc.bf16_round(m - tol)).astype(np.float64)
        hi = wl.bf16_to_f32(orc.bf16_round(m + tol)).astype(np.float64)
        ok = (lo <= g) & (g <= hi)
        assert np.all(ok), f"{int((~ok).sum())} z elements off beyond the fp32 error"
    print(f"[audio head] z: {n} of {z_gpu.size} roundings taken the other way within the fp32 error")


CASES = [
    # (R, H, F, V, n_tail, mode, T)
    (5, 128, 256, 300, 3, "argmax", 0.0),            # ragged rows, a 3-id tail
    (64, 2048, 4096, 4097, 1, "argmax", 0.0),        # an acoustic stage (4,096 codes + boundary)
    (16, 2048, 4096, 16386, 2, "argmax", 0.0),       # CB0: 16,384 codes + row terminator + <|audio_split|>
    (16, 2048, 4096, 16386, 2, "gumbel", 0.7),
    (40, 512, 1024, 777, 0, "gumbel", 1.3),          # no structural tail
    (160, 256, 512, 1000, 3, "argmax", 0.0),         # 160 rows: the wide argmax build, with tail masks and bias
]


@pytest.mark.parametrize("case", CASES, ids=[f"R{c[0]}-F{c[2]}-V{c[3]}-{c[5]}" for c in CASES])
def test_audio_head_matches_oracle(orc, bd, case):
    R, H, F, V, n_tail, mode, T = case
    inp = wl.audio_head_inputs(R, H, F, V, n_tail, seed=3000 + CASES.index(case))
    z_ref, mish_ref = orc.audio_expand(inp["h"], inp["W1"], inp["b1"])
    ref = orc.head_select_masked(z_ref, inp["W2"], inp["b2"], mode, T, inp["seed"], inp["step"], n_tail,
                                 inp["tail_allowed"], want_logits=True)
    z, ids, best, logits = _run(bd, inp, R, F, V, n_tail, mode, T, logits=True)
    check_z(orc, inp, z, z_ref, mish_ref)
    err = np.abs(logits.astype(np.float64) - ref["logits"])
    assert err.max() <= 2e-3, f"logits differ by {err.max():.3g}"
    hard, ties = compare_ids(ids, ref)
    print(f"[audio head {case}] logits max abs err {err.max():.2g}; near-ties {ties}, hard mismatches {len(hard)}")
    assert not hard
    # a chosen tail id is always allowed for its row
    for r in range(R):
        j = int(ids[r]) - (V - n_tail)
        if n_tail and j >= 0:
            assert (int(inp["tail_allowed"][r]) >> j) & 1


@pytest.mark.parametrize("case", [c for c in CASES if c[0] <= 64],
                         ids=[f"R{c[0]}-F{c[2]}-V{c[3]}-{c[5]}" for c in CASES if c[0] <= 64])
def test_audio_head_ids_without_logits(orc, bd, case):
    """The same heads without the logits written out: narrow batches then
    select in the split build (bias, tail masks and Gumbel noise included)."""
    R, H, F, V, n_tail, mode, T = case
    inp = wl.audio_head_inputs(R, H, F, V, n_tail, seed=3000 + CASES.index(case))
    z_ref, _ = orc.audio_expand(inp["h"], inp["W1"], inp["b1"])
    z, ids, best, _ = _run(bd, inp, R, F, V, n_tail, mode, T, logits=False)
    # the second layer selects over the GPU's own z (exact inputs)
    ref = orc.head_select_masked(z, inp["W2"], inp["b2"], mode, T, inp["seed"], inp["step"], n_tail,
                                 inp["tail_allowed"])
    hard, ties = compare_ids(ids, ref)
    assert not hard, f"rows {hard[:10]} (near-ties {ties})"


def test_audio_head_tail_mask_decides(orc, bd):
    """Structural ids made dominant by their bias win exactly where their bit
    is set: the highest allowed tail id, else the codebook's argmax."""
    R, H, F, V, n_tail = 24, 256, 512, 1000, 3
    inp = wl.audio_head_inputs(R, H, F, V, n_tail, seed=3100)
    inp["b2"][V - n_tail:] = [50.0, 60.0, 70.0]
    inp["tail_allowed"] = np.arange(R, dtype=np.uint32) % 8
    z_ref, _ = orc.audio_expand(inp["h"], inp["W1"], inp["b1"])
    ref = orc.head_select_masked(z_ref, inp["W2"], inp["b2"], "argmax", 0.0, None, None, n_tail,
                                 inp["tail_allowed"])
    _, ids, _, _ = _run(bd, inp, R, F, V, n_tail)
    for r in range(R):
        m = int(inp["tail_allowed"][r])
        if m:
            assert ids[r] == V - n_tail + m.bit_length() - 1
        else:
            assert ids[r] < V - n_tail
    hard, _ = compare_ids(ids, ref)
    assert not hard
    # no mask: every tail id allowed, the largest bias wins everywhere
    _, ids_all, _, _ = _run(bd, inp, R, F, V, n_tail, masked=False)
    assert np.all(ids_all == V - 1)


def test_audio_head_rejects_bad_shapes(bd):
    R, H, F, V = 4, 128, 256, 300
    inp = wl.audio_head_inputs(R, H, F, V, 1, seed=5)
    ws = torch.zeros(bd.tts_head_workspace_size(R, V), dtype=torch.uint8, device="cuda")
    ids = torch.empty(R, dtype=torch.int32, device="cuda")
    args = (dev(inp["h"]), dev(inp["W1"]), None, dev(inp["W2"]), None)
    z = torch.empty((R, F), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bd.TTSError) as e:
        bd.tts_audio_head_select(*args, z, ids, ws, n_tail=33)
    assert e.value.code == ERR_INVALID
    # F not a multiple of 64
    inp2 = wl.audio_head_inputs(R, H, 200, V, 1, seed=6)
    z2 = torch.empty((R, 200), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bd.TTSError) as e:
        bd.tts_audio_head_select(dev(inp2["h"]), dev(inp2["W1"]), None, dev(inp2["W2"]), None, z2, ids, ws)
    assert e.value.code == ERR_UNSUPPORTED
    # Gumbel without keys
    with pytest.raises(bd.TTSError) as e:
        bd.tts_audio_head_select(*args, z, ids, ws, mode=bd.TTS_GUMBEL, temperature=0.7)
    assert e.value.code == ERR_INVALID
