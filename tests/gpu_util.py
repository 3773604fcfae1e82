"""Helpers for the GPU parity tests: upload generated inputs, run the oracle,
compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import workloads as wl

# Attention: element passes when |gpu - oracle| <= max(ATOL, RTOL * |oracle|).
ATOL, RTOL = 2e-2, 1e-2
# Token choices: a mismatch is allowed only where the oracle's top two keys
# (or acceptance ratio and uniform) are closer than this.
NEAR_TIE = 1e-3


def dev(x: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays holding bf16 bits become bfloat16."""
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    if x.dtype == np.uint64:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int64)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> numpy; bfloat16 comes back as uint16 bits."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    return wl.to_f32(x, dtype).astype(np.float64)


def attn_errors(gpu: np.ndarray, ref: np.ndarray):
    """(number of failing elements, max abs error, max rel error over |ref| >= ATOL)."""
    err = np.abs(gpu - ref)
    bound = np.maximum(ATOL, RTOL * np.abs(ref))
    bad = int((~(err <= bound)).sum())
    big = np.abs(ref) >= ATOL
    rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return bad, float(err.max()) if err.size else 0.0, rel


def rel_where_binding(gpu: np.ndarray, ref: np.ndarray) -> float:
    """Max relative error over the elements where the relative bound is the
    larger one (|ref| >= ATOL / RTOL); 0 if there are none."""
    big = np.abs(ref) >= ATOL / RTOL
    return float((np.abs(gpu - ref)[big] / np.abs(ref[big])).max()) if big.any() else 0.0


def compare_ids(gpu_ids, ref, near=NEAR_TIE):
    """Mismatched rows that are not near-ties, and the near-tie count."""
    gap = ref["best"].astype(np.float64) - ref["second"].astype(np.float64)
    tie = gap < near
    mism = np.nonzero(gpu_ids != ref["ids"])[0]
    hard = [int(r) for r in mism if not tie[r]]
    return hard, int(tie.sum())


class Uploaded:
    """Device copies of one workload's inputs."""

    def __init__(self, inp: dict):
        self.inp = inp
        self.w = inp["workload"]
        self.table = dev(inp["block_table"])
        self.ctx_before = dev(inp["ctx_before"])
        self.ctx_lens = dev(inp["ctx_lens"])
        self.k_pool = dev(inp["k_pool"])
        self.v_pool = dev(inp["v_pool"])
        self.q = dev(inp["q"])
        self.k_new = dev(inp["k_new"])
        self.v_new = dev(inp["v_new"])
        for k in ("h", "W", "seed", "step", "target_logits", "draft_probs", "draft_tokens",
                  "vseed", "vstep"):
            if k in inp:
                setattr(self, k, dev(inp[k]))
