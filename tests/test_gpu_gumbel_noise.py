"""The Gumbel noise of every Gumbel-max draw on the device: the head's seeded
Gumbel-top-1 draw at temperature T, the code predictor's, and the speculative
verify's residual and bonus draws ("Optimizing Streaming Text-to-Speech Models
for Sub-50 Millisecond Latency", section "Speculative Decoding for Acoustic
Tokens").  The kernels evaluate -ln(-ln u) with a Taylor series of
-ln(1 - w) near u = 1 and the hardware base-2 logarithm elsewhere; this test
evaluates it on the device for every one of the 2^23 values u = (2k + 1) / 2^24
the Philox words map to and bounds its distance to the exact value (float64).
The bound is far below the 1e-3 within which the draw's keys count as
near-ties."""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BOUND = 1e-5


def test_gumbel_noise_within_bound_for_every_uniform(parity):
    from decode_step_gb300 import binding as bd
    k = np.arange(1 << 23, dtype=np.uint32)
    bits = torch.from_numpy((k << np.uint32(9)).view(np.int32)).cuda()
    out = torch.empty(k.size, dtype=torch.float32, device="cuda")
    bd.tts_test_gumbel_noise(bits, out)
    torch.cuda.synchronize()
    u = (2.0 * k.astype(np.float64) + 1.0) / 2.0 ** 24
    exact = -np.log(-np.log(u))
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - exact)
    worst = int(np.argmax(err))
    parity("Gumbel noise vs exact", values=int(k.size), max_abs=float(err.max()))
    assert err.max() <= BOUND, f"max |error| {err.max():.3e} at u = {u[worst]!r}"

