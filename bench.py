#!/usr/bin/env python
"""Benchmark of one batched decode step (append -> attention -> head) on GB300.

Workload (default): 64 streams, GQA 16 query / 8 KV heads, head_dim 128, bf16,
context lengths uniform in [50, 1500] behind a randomly permuted block table,
acoustic head 2048 -> 4097 at temperature zero.  A step processes one query
token per stream; value = codec tokens per second = streams / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Prints one JSON line.  Under torchrun (N > 1) every rank runs its own replica
of the workload on its own GPU (streams are independent; no collective on the
data path); timing is the max over ranks.  --impl reference times the CPU
oracle on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "codec tokens/s per decode batch; decode-attn HBM GB/s and % of GB300 peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
ATTN_SOURCES = ["decode_step_gb300/csrc/decode_attn.cu", "decode_step_gb300/csrc/tts_common.cuh"]


# ------------------------------------------------------------------ helpers

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", type=int, default=3, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work budget of the oracle baseline in the native line")
    ap.add_argument("--e2e-steps", type=int, default=1000)
    ap.add_argument("--e2e-sizes", default="1,4,16,64",
                    help="active-stream counts timed end to end through the captured-step set ('' for none)")
    ap.add_argument("--sweep", default="2,4,5,3f",
                    help="other workloads whose kernels are timed one by one into the line's "
                         "'workloads' object (comma-separated ids, 'f' suffix: FP8 E4M3 KV cache; "
                         "empty: none)")
    ap.add_argument("--sweep-reps", type=int, default=30)
    ap.add_argument("--chained", type=int, default=1,
                    help="time the kernels back to back as programmatic dependents (needs a second copy of "
                         "the cache and 15 more of W; 0 to skip, e.g. for profiling runs)")
    ap.add_argument("--code-predictor", type=int, default=1,
                    help="time the code predictor's frame loop (workloads.CODE_PREDICTOR; 0 to skip)")
    ap.add_argument("--audio-heads", default="acoustic-b64,semantic-cb0-b16",
                    help="two-layer audio-head shapes timed alone (names of workloads.AUDIO_HEAD_SHAPES; '' for none)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def combine_rank_times(per_rank_ms: list[float], streams_per_rank: int) -> tuple[float, float]:
    """(ms per step = max over ranks, whole-job tokens/s = all ranks' streams / that time)."""
    ms = max(per_rank_ms)
    return ms, streams_per_rank * len(per_rank_ms) / (ms / 1e3)


def max_over_ranks(x: float, world: int, device=None) -> list[float]:
    """All ranks' values of x (gathered; works for nccl and gloo groups)."""
    if world == 1:
        return [x]
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return [float(o.item()) for o in out]


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        h.update((ROOT / p).read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the capture (else None)."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    try:
        rec = json.loads(p.read_text()).get(kernel)
    except (ValueError, AttributeError):
        return None
    if not rec or rec.get("workload") != workload or rec.get("source_sha") != source_sha(ATTN_SOURCES):
        return None
    return rec.get("dram_bytes_per_launch")


def attn_bytes(inp) -> int:
    """Algorithmic bytes of one attention launch: every cached K/V row once,
    q and out once, the used block-table entries and the context lengths."""
    w = inp["workload"]
    L = inp["ctx_lens"].astype(np.int64)
    kv = int(L.sum()) * w.Hkv * w.D * w.elem_bytes * 2
    qo = 2 * w.B * w.q_len * w.Hq * w.D * w.elem_bytes
    table = int((-(-L // wl.BLOCK)).sum()) * 4
    return kv + qo + table + 4 * w.B


def attn_bytes_fp8(inp) -> int:
    """Algorithmic bytes of one attention launch over an FP8 cache: every
    cached key and value row once as codes plus its fp32 scale (4224 bytes per
    16 tokens and KV head), q and out (bf16), the used block-table entries and
    the context lengths."""
    w = inp["workload"]
    L = inp["ctx_lens"].astype(np.int64)
    kv = int(L.sum()) * w.Hkv * (w.D + 4) * 2
    qo = 2 * w.B * w.q_len * w.Hq * w.D * 2
    table = int((-(-L // wl.BLOCK)).sum()) * 4
    return kv + qo + table + 4 * w.B


def head_bytes(w) -> int:
    return w.V * w.H * w.elem_bytes + w.R * w.H * w.elem_bytes + 4 * w.R


def head_line_bytes(w) -> int:
    """Head bytes including the fp32 logits the verify path writes out."""
    return head_bytes(w) + (w.R * w.V * 4 if w.logits_out else 0)


def verify_bytes(w) -> int:
    """Algorithmic bytes of one spec-verify launch without the bonus draw: the
    K target rows and K draft rows of every stream (fp32), the draft tokens,
    the two outputs."""
    return 2 * w.B * w.K * w.V * 4 + w.B * w.K * 4 + 2 * w.B * 4


def append_bytes(w) -> int:
    return 2 * 2 * w.B * w.q_len * w.Hkv * w.D * w.elem_bytes


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.25)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in Path(self.path).read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle

def oracle_stream_steps(orc, inp, streams, kp, vp, keep=None):
    """The oracle's decode step for a list of streams (append, attention, head
    row).  keep (a dict, optional) receives stream -> (attention output, head
    result) of the streams run."""
    w = inp["workload"]
    for b in streams:
        sl = slice(b, b + 1)
        orc.kv_append(kp, vp, inp["block_table"][sl], inp["ctx_before"][sl], inp["k_new"][sl],
                      inp["v_new"][sl], inplace=True)
        att = orc.decode_attn(kp, vp, inp["block_table"][sl], inp["ctx_lens"][sl], inp["q"][sl],
                              inp["scale"], w.causal)
        h = wl.f32_to_bf16(att.reshape(w.q_len, -1).astype(np.float32)) if w.dtype == "bf16" \
            else att.reshape(w.q_len, -1).astype(np.float32)
        res = orc.head_select(h, inp["W"], w.mode, w.T, inp["seed"][b * w.q_len:(b + 1) * w.q_len],
                              inp["step"][b * w.q_len:(b + 1) * w.q_len])
        if keep is not None:
            keep[b] = (att, res)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_throughput(orc, inp, seconds: float, threads: int, keep=None) -> tuple[float, int]:
    """Stream-steps per second of the oracle over about `seconds` of wall time:
    `threads` Python threads (the oracle is C behind ctypes, which releases
    the interpreter lock) each cycling over its own share of the streams
    (thread t takes streams t, t + threads, ...), all writing one copy of the
    pool (every stream appends to its own slots).  Returns (stream-steps/s,
    stream-steps run)."""
    import threading
    w = inp["workload"]
    kp, vp = inp["k_pool"].copy(), inp["v_pool"].copy()
    counts = [0] * threads
    stop = time.perf_counter() + seconds

    def work(t):
        mine = list(range(t, w.B, threads)) or [t % w.B]
        i = 0
        while counts[t] == 0 or time.perf_counter() < stop:
            b = mine[i % len(mine)]
            oracle_stream_steps(orc, inp, [b], kp, vp, keep if (keep is not None and i < len(mine)) else None)
            counts[t] += 1
            i += 1

    t0 = time.perf_counter()
    if threads == 1:
        work(0)
    else:
        pool = [threading.Thread(target=work, args=(t,)) for t in range(threads)]
        for th in pool:
            th.start()
        for th in pool:
            th.join()
    dt = time.perf_counter() - t0
    return sum(counts) * w.q_len / dt, sum(counts)


def parity_against(inp, keep, gpu_out, gpu_ids) -> dict:
    """The GPU step's attention output and ids against the oracle's, for the
    streams the CPU baseline ran (attention: max-abs / max-rel and elements
    outside max(2e-2, 1e-2 |o|); ids: near-ties, where the oracle's top two
    keys are closer than 1e-3, and mismatches outside them)."""
    w = inp["workload"]
    if not keep:
        return {}
    mx_abs = mx_rel = 0.0
    bad = elements = ties = hard = 0
    for b, (att, res) in keep.items():
        g = gpu_out[b].astype(np.float64)
        err = np.abs(g - att)
        bad += int((~(err <= np.maximum(2e-2, 1e-2 * np.abs(att)))).sum())
        elements += att.size
        mx_abs = max(mx_abs, float(err.max()))
        big = np.abs(att) >= 2e-2
        if big.any():
            mx_rel = max(mx_rel, float((err[big] / np.abs(att[big])).max()))
        gid = gpu_ids[b * w.q_len:(b + 1) * w.q_len]
        tie = (res["best"].astype(np.float64) - res["second"].astype(np.float64)) < 1e-3
        ties += int(tie.sum())
        hard += int(((gid != res["ids"]) & ~tie).sum())
    return {"streams": len(keep), "attention_max_abs": mx_abs, "attention_max_rel": mx_rel,
            "attention_outside_tolerance": bad, "attention_elements": elements, "id_rows": len(keep) * w.q_len,
            "id_near_ties": ties, "id_mismatches_outside_near_ties": hard,
            "note": "the step's GPU outputs against the oracle for the streams the CPU baseline ran"}


def cpu_baseline(inp, seconds: float, gpu_out=None, gpu_ids=None) -> tuple[dict, dict]:
    """The oracle over whole stream-steps (append, attention, head row) of this
    workload: single-threaded for half of `seconds`, then one thread per host
    core (os.sched_getaffinity) for the other half.  Returns (cpu_baseline,
    parity of the GPU outputs for the streams run single-threaded)."""
    import oracle
    orc = oracle.default()
    w = inp["workload"]
    keep = {} if gpu_out is not None else None
    v1, n1 = oracle_throughput(orc, inp, seconds / 2, 1, keep)
    cores = host_cores()
    vn, nn = oracle_throughput(orc, inp, seconds / 2, cores)
    base = {"value": vn, "unit": UNIT, "cores": cores, "kind": "oracle",
            "single_thread_value": v1,
            "sample": f"stream-steps (append, attention, head row) cycling over the {w.B} streams of one step: "
                      f"{nn} on {cores} threads (one per host core in the affinity mask) and {n1} single-threaded, "
                      f"about {seconds / 2:.0f} s each; C oracle"}
    par = parity_against(inp, keep, gpu_out, gpu_ids) if keep is not None else {}
    return base, par


# ------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import threading
    import oracle
    orc = oracle.default()
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w)
    kp, vp = inp["k_pool"].copy(), inp["v_pool"].copy()
    cores = host_cores()
    # One unit = one stream's step; a step of this arm is a bounded sample of
    # units (spread over one thread per host core) sized so that warm-up +
    # timed steps take about two minutes.
    t0 = time.perf_counter()
    oracle_stream_steps(orc, inp, [0], kp, vp)
    unit_s = max(time.perf_counter() - t0, 1e-4)
    per_step = max(1, min(w.B, int(cores * 120.0 / (args.steps + args.warmup) / unit_s)))
    order = np.random.default_rng(0).permutation(w.B)
    pos = 0

    def one_step():
        nonlocal pos
        streams = [int(order[(pos + i) % w.B]) for i in range(per_step)]
        pos += per_step
        n = min(cores, len(streams))
        parts = [streams[t::n] for t in range(n)]
        ths = [threading.Thread(target=oracle_stream_steps, args=(orc, inp, part, kp, vp)) for part in parts]
        for th in ths:
            th.start()
        for th in ths:
            th.join()

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = time.perf_counter() - t0
    tokens = per_step * w.q_len * args.steps
    value = tokens / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} of {w.B} streams per step, split over {min(cores, per_step)} threads "
                                   f"(one per host core in the affinity mask), C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def kernel_sweep(ids, reps, flush_l2, peaks, device) -> dict:
    """Each kernel of the other workloads launched alone `reps` times, L2
    flushed before every launch, CUDA events around it (mean over launches),
    with its roofline fraction against the measured HBM peak (tensor peak too
    for the head).  The pool is appended to once first, so attention reads
    the step's own new tokens."""
    import torch
    from decode_step_gb300 import binding as bd

    def dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        if x.dtype == np.uint64:
            return torch.from_numpy(x.view(np.int64)).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    def timed(fn):
        ts = []
        for _ in range(reps):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.fmean(ts[2:])

    hbm = peaks["hbm_gbs"]
    out = {}
    for wid in ids:
        fp8 = str(wid).endswith("f")
        w = wl.WORKLOADS[int(str(wid).rstrip("f"))]
        inp = wl.make_inputs(w)
        d = {k: dev(inp[k]) for k in ("block_table", "ctx_before", "ctx_lens", "q", "k_new", "v_new", "h", "W",
                                       "seed", "step")}
        if fp8:
            # the context quantised by the library's own append, one stream at a time
            kp, vp = dev(inp["k_pool"]), dev(inp["v_pool"])
            nb = kp.shape[0]
            cache = bd.KVCache(torch.zeros((nb, w.Hkv, bd.KVCache.FP8_TILE_BYTES), dtype=torch.uint8, device=device))
            zero = torch.zeros(1, dtype=torch.int32, device=device)
            for b in range(w.B):
                n = int(inp["ctx_before"][b])
                if n == 0:
                    continue
                t = torch.arange(n, device=device)
                blocks = d["block_table"][b, t // wl.BLOCK].long()
                rows_k = kp[blocks, :, t % wl.BLOCK, :].unsqueeze(0).contiguous()
                rows_v = vp[blocks, :, t % wl.BLOCK, :].unsqueeze(0).contiguous()
                bd.tts_kv_append(cache, d["block_table"][b:b + 1].contiguous(), zero, rows_k, rows_v)
            del kp, vp
        else:
            cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
        bd.tts_kv_append(cache, d["block_table"], d["ctx_before"], d["k_new"], d["v_new"])
        attn_out = torch.empty_like(d["q"])
        ws = torch.zeros(bd.tts_decode_attn_workspace_size(w.B, w.q_len, w.Hq, w.Hkv, w.D, w.ctx_hi),
                         dtype=torch.uint8, device=device)
        t_att = timed(lambda: bd.tts_decode_attn(cache, d["block_table"], d["ctx_lens"], w.ctx_hi, d["q"],
                                                 attn_out, ws, inp["scale"], w.causal))
        ab = attn_bytes_fp8(inp) if fp8 else attn_bytes(inp)
        ids_t = torch.empty(w.R, dtype=torch.int32, device=device)
        hws = torch.zeros(bd.tts_head_workspace_size(w.R, w.V), dtype=torch.uint8, device=device)
        logits = torch.empty(w.R, w.V, dtype=torch.float32, device=device) if w.logits_out else None
        mode = bd.TTS_GUMBEL if w.mode == "gumbel" else bd.TTS_ARGMAX
        t_head = timed(lambda: bd.tts_codebook_head_select(d["h"], d["W"], ids_t, hws, mode=mode,
                                                           temperature=w.T, seed=d["seed"], step=d["step"],
                                                           logits_out=logits))
        hb = head_line_bytes(w)
        flops = 2.0 * w.R * w.H * w.V
        entry = {
            "decode_attn_us": t_att, "decode_attn_gbs": ab / t_att / 1e3, "decode_attn_frac": ab / t_att / 1e3 / hbm,
            "decode_attn_bytes": ab,
            "head_select_us": t_head, "head_gbs": hb / t_head / 1e3, "head_frac_hbm": hb / t_head / 1e3 / hbm,
            "head_tflops": flops / t_head / 1e6,
            "head_frac_tensor": flops / t_head / 1e6 / peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]),
            "head_bytes": hb, "head_mode": w.mode, "kv_cache": "fp8_e4m3" if fp8 else w.dtype,
        }
        # the append alone, plain and with the rotary embedding of q and k_new
        # (q rotated in place again on every launch: only its timing is used)
        entry["kv_append_us"] = timed(lambda: bd.tts_kv_append(cache, d["block_table"], d["ctx_before"],
                                                               d["k_new"], d["v_new"]))
        entry["kv_append_rope_us"] = timed(lambda: bd.tts_kv_append_rope(cache, d["block_table"], d["ctx_before"],
                                                                         d["q"], d["k_new"], d["v_new"]))
        if fp8:
            from decode_step_gb300.step import DecodeStep
            kw = dict(q_len=w.q_len, causal=w.causal, mode=bd.TTS_GUMBEL if w.mode == "gumbel" else bd.TTS_ARGMAX,
                      temperature=w.T)
            stp = DecodeStep(cache, d["W"], w.Hq, w.B, w.ctx_hi, **kw)
            stp_rope = DecodeStep(cache, d["W"], w.Hq, w.B, w.ctx_hi, rope_base=10000.0, **kw)
            t_step = timed(lambda: stp(d["block_table"], d["ctx_before"], d["ctx_lens"], d["q"], d["k_new"],
                                       d["v_new"], seed=d["seed"], step=d["step"]))
            t_rope = timed(lambda: stp_rope(d["block_table"], d["ctx_before"], d["ctx_lens"], d["q"], d["k_new"],
                                            d["v_new"], seed=d["seed"], step=d["step"]))
            entry.update({"step_us": t_step, "tokens_per_s": w.B * w.q_len / (t_step * 1e-6),
                          "step_rope_us": t_rope, "tokens_per_s_rope": w.B * w.q_len / (t_rope * 1e-6)})
        if w.K > 0:
            tl, dp = dev(inp["target_logits"]), dev(inp["draft_probs"])
            dt, vs, vt = dev(inp["draft_tokens"]), dev(inp["vseed"]), dev(inp["vstep"])
            n_acc = torch.empty(w.B, dtype=torch.int32, device=device)
            nxt = torch.empty(w.B, dtype=torch.int32, device=device)
            t_ver = timed(lambda: bd.tts_spec_verify(tl, dp, dt, w.T, vs, vt, n_acc, nxt))
            vb = verify_bytes(w)
            # with the launch latency hidden: 32 launches over 16 copies of the
            # rows (beyond L2) captured as one graph, each a programmatic
            # dependent of the one before, replayed 8 times between events
            vsets = [(tl, dp)] + [(tl.clone(), dp.clone()) for _ in range(15)]
            for i in range(4):
                bd.tts_spec_verify(*vsets[i % 16], dt, w.T, vs, vt, n_acc, nxt)
            prev = bd.tts_set_launch_flags(bd._lib.LAUNCH_PROGRAMMATIC)
            try:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, capture_error_mode="thread_local"):
                    for i in range(32):
                        bd.tts_spec_verify(*vsets[i % 16], dt, w.T, vs, vt, n_acc, nxt)
            finally:
                bd.tts_set_launch_flags(prev)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(8):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            t_ver_chain = e0.elapsed_time(e1) * 1e3 / (8 * 32)
            del g, vsets
            entry.update({"spec_verify_us": t_ver, "spec_verify_gbs": vb / t_ver / 1e3,
                          "spec_verify_frac": vb / t_ver / 1e3 / hbm, "spec_verify_bytes": vb,
                          "spec_verify_us_chained": t_ver_chain,
                          "spec_verify_frac_chained": vb / t_ver_chain / 1e3 / hbm})
            # the whole speculative step captured once (inputs from pinned
            # memory, append, causal attention over K + 1 rows, Gumbel head
            # keeping its logits, verify, results to pinned memory): wall
            # clock per step, synchronised every step
            from decode_step_gb300.step import DecodeStep, GraphedStep
            vstep_ = DecodeStep(cache, d["W"], w.Hq, w.B, w.ctx_hi, q_len=w.q_len, causal=w.causal,
                                mode=bd.TTS_GUMBEL, temperature=w.T)
            gin = {k: d[k] for k in ("block_table", "ctx_before", "ctx_lens", "q", "k_new", "v_new", "seed", "step")}
            gin.update({"draft_probs": dp, "draft_tokens": dt, "vseed": vs, "vstep": vt})
            gv = GraphedStep(vstep_, gin, verify_temperature=w.T)
            for _ in range(5):
                gv()
            t0 = time.perf_counter()
            for _ in range(reps * 4):
                gv()
            us = (time.perf_counter() - t0) / (reps * 4) * 1e6
            entry.update({"verify_step_e2e_us": us,
                          "verify_step_note": "captured step with verify, host sync per step; each stream "
                                              "advances 1 + accepted tokens"})
            del gv, vstep_
        out[w.name + ("-fp8" if fp8 else "")] = entry
        del cache, d, attn_out, ws
        torch.cuda.empty_cache()
    return out


def audio_head_bytes(R, H, F, V) -> int:
    """Algorithmic bytes of one two-layer audio head: both weight matrices and
    biases once, h, z written by the first layer and read by the second, the
    row masks and the ids."""
    return 2 * F * H + 4 * F + 2 * V * F + 4 * V + 2 * R * H + 2 * (2 * R * F) + 4 * R + 4 * R


def audio_head_sweep(names, reps, flush_l2, peaks, device) -> dict:
    """tts_audio_head_select (expansion + Mish, then the masked head) launched
    alone `reps` times, L2 flushed before each, CUDA events around the call."""
    import torch
    from decode_step_gb300 import binding as bd

    def dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        if x.dtype in (np.uint64, np.uint32):
            return torch.from_numpy(x.view(np.int64 if x.dtype == np.uint64 else np.int32)).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    out = {}
    for name in names:
        R, H, F, V, n_tail = wl.AUDIO_HEAD_SHAPES[name]
        inp = wl.audio_head_inputs(R, H, F, V, n_tail)
        d = {k: dev(v) for k, v in inp.items()}
        z = torch.empty((R, F), dtype=torch.bfloat16, device=device)
        ids = torch.empty(R, dtype=torch.int32, device=device)
        ws = torch.zeros(bd.tts_head_workspace_size(R, V), dtype=torch.uint8, device=device)
        res = {}
        for mode in ("argmax", "gumbel"):
            m = bd.TTS_GUMBEL if mode == "gumbel" else bd.TTS_ARGMAX

            def call():
                bd.tts_audio_head_select(d["h"], d["W1"], d["b1"], d["W2"], d["b2"], z, ids, ws, mode=m,
                                         temperature=0.7, seed=d["seed"], step=d["step"], n_tail=n_tail,
                                         tail_allowed=d["tail_allowed"])
            ts = []
            for _ in range(reps):
                flush_l2()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                call()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
            t = statistics.fmean(ts[2:])
            nb = audio_head_bytes(R, H, F, V)
            res[mode] = {"us": t, "gbs": nb / t / 1e3, "frac_hbm": nb / t / 1e3 / peaks["hbm_gbs"], "bytes": nb,
                         "tflops": 2.0 * R * (H * F + F * V) / t / 1e6}
        out[name] = {"shape": {"R": R, "H": H, "F": F, "V": V, "n_tail": n_tail}, **res}
        del d, z, ids, ws
        torch.cuda.empty_cache()
    return out


def predictor_bytes(R, H, Hq, Hkv, D, V, n_steps) -> int:
    """Algorithmic bytes of one frame of the code predictor: the projection
    weights once (they stay in L2 across the steps), every codebook head once,
    the gathered embedding rows, the talker states, the cache rows written and
    read, and the tokens."""
    F = (Hq + 2 * Hkv) * D
    return (2 * F * H + 2 * n_steps * V * H + 2 * (n_steps - 1) * R * H + 2 * R * H
            + 2 * n_steps * R * 2 * Hkv * D * 2 + 4 * n_steps * R)


def predictor_sweep(reps, flush_l2, peaks, device) -> dict:
    """The frame loop for workloads.CODE_PREDICTOR: the persistent kernel
    (launched, and captured with its control-word reset) and the
    kernel-per-stage graph; L2 flushed before each run, CUDA events around it."""
    import torch
    from decode_step_gb300 import binding as bd
    c = wl.CODE_PREDICTOR
    R, H, Hq, Hkv, D, V, n = c["R"], c["H"], c["Hq"], c["Hkv"], c["D"], c["V"], c["n_steps"]
    inp = wl.code_predictor_inputs(R, H, Hq, Hkv, D, V, n)

    def dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(x.view(np.int64) if x.dtype == np.uint64 else x).to(device)

    args = [dev(inp[k]) for k in ("x0", "Wqkv", "W", "E")]
    tokens = torch.empty((n, R), dtype=torch.int32, device=device)
    nb = predictor_bytes(R, H, Hq, Hkv, D, V, n)
    out = {"shape": dict(c), "bytes": nb,
           "kernels_per_frame": {"persistent": 1, "multi_kernel": 1 + 5 * n - 1}}
    for kind in ("persistent", "persistent_graph", "multi_kernel_graph"):
        cp = bd.CodePredictor(*args, Hq, Hkv, tokens, graph=kind.endswith("graph"),
                              multi_kernel=kind.startswith("multi"))
        for _ in range(3):
            cp.run()
        ts = []
        for _ in range(reps):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            cp.run()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        t = statistics.fmean(ts[2:])
        out[kind] = {"us_per_frame_batch": t, "frames_per_s": R / (t * 1e-6), "tokens_per_s": R * n / (t * 1e-6),
                     "gbs": nb / t / 1e3, "frac_hbm": nb / t / 1e3 / peaks["hbm_gbs"]}
        cp.close()
    return out


def workload_config(w, world):
    return {"workload": f"{w.name}: {w.B} streams/GPU, GQA {w.Hq}/{w.Hkv} heads, head_dim {w.D}, "
                        f"{w.dtype}, q_len {w.q_len}, ctx {w.ctx_dist} [{w.ctx_lo},{w.ctx_hi}], "
                        f"{'permuted' if w.permute_table else 'ordered'} 16-token block table, "
                        f"head {w.H}->{w.V} {w.mode}",
            "global_batch": w.B * world, "seq_len": 1, "l2": "flushed before every timed step: a 2x-L2 buffer written, then another read",
            "parallelism": f"replicas x{world} (streams independent, no collective)"}


# ---------------------------------------------------------------- native arm

def run_native(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    from decode_step_gb300.build import build as build_lib
    build_lib()
    from decode_step_gb300 import binding as bd
    from decode_step_gb300.step import DecodeStep

    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w, seed=wl.NUMPY_SEED_BASE + w.id + 7919 * rank)

    def dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        if x.dtype == np.uint64:
            return torch.from_numpy(x.view(np.int64)).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    names = ["block_table", "ctx_before", "ctx_lens", "q", "k_new", "v_new"]
    d = {k: dev(inp[k]) for k in names}
    seed, stp = dev(inp["seed"]), dev(inp["step"])
    cache = bd.KVCache(dev(inp["k_pool"]), dev(inp["v_pool"]))
    W = dev(inp["W"])
    mode = bd.TTS_GUMBEL if w.mode == "gumbel" else bd.TTS_ARGMAX
    step = DecodeStep(cache, W, w.Hq, w.B, w.ctx_hi, q_len=w.q_len, causal=w.causal, mode=mode,
                      temperature=w.T)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    # L2 flush between timed steps: write a buffer twice the L2 size, then read
    # another one as large.  The write alone evicts the step's inputs but
    # leaves the L2 full of dirty lines whose write-back then lands inside the
    # next timed kernel (about 10 us on a 200 MB read); the read evicts them
    # outside the timed region, so every step starts cold and clean, the state
    # a serving loop leaves (its steps write a few hundred KB).  The per-kernel
    # pass also reports the write-only figures.
    n_flush = max(2 * l2, 256 << 20)
    flush = torch.empty(n_flush, dtype=torch.uint8, device=device)
    flush_read = torch.ones(n_flush, dtype=torch.uint8, device=device)

    def flush_l2(write_only: bool = False):
        flush.zero_()
        if not write_only:
            torch.amax(flush_read)

    stream = torch.cuda.current_stream()

    def run_step():
        return step(d["block_table"], d["ctx_before"], d["ctx_lens"], d["q"], d["k_new"],
                    d["v_new"], seed=seed, step=stp)

    for _ in range(max(args.warmup, 3)):
        flush_l2()
        run_step()
    torch.cuda.synchronize()

    # ---- timed region: K whole steps (one tts_decode_step call each: append,
    # attention and head, the later two as programmatic dependents), L2
    # flushed before every step outside the events.
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2()
        ev[i][0].record(stream)
        run_step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    t_step = [e[0].elapsed_time(e[1]) for e in ev]
    ms_local = statistics.fmean(t_step)
    all_ms = max_over_ranks(ms_local, world, device)
    ms, value = combine_rank_times(all_ms, w.B * w.q_len)
    errflags = int(step.err.item())

    # ---- per-kernel durations: the same kernels launched one by one, each
    # bracketed by events (no overlap between them), L2 flushed per step.
    K2 = min(K, 1000)
    K3 = min(K2, 200)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K2 + K3)]
    for i in range(K2 + K3):
        flush_l2(write_only=i >= K2)
        e = kev[i]
        e[0].record(stream)
        bd.tts_kv_append(cache, d["block_table"], d["ctx_before"], d["k_new"], d["v_new"], err=step.err)
        e[1].record(stream)
        bd.tts_decode_attn(cache, d["block_table"], d["ctx_lens"], w.ctx_hi, d["q"], step.out,
                           step.attn_ws, step.scale, w.causal, err=step.err)
        e[2].record(stream)
        bd.tts_codebook_head_select(step.out.view(step.R, -1), W, step.ids, step.head_ws, mode=mode,
                                    temperature=w.T, seed=seed, step=stp)
        e[3].record(stream)
    torch.cuda.synchronize()
    t_app = [e[0].elapsed_time(e[1]) for e in kev[:K2]]
    t_att = [e[1].elapsed_time(e[2]) for e in kev[:K2]]
    t_head = [e[2].elapsed_time(e[3]) for e in kev[:K2]]
    t_att_w = [e[1].elapsed_time(e[2]) for e in kev[K2:]]
    t_head_w = [e[2].elapsed_time(e[3]) for e in kev[K2:]]

    # ---- per-kernel durations with the launch latency hidden, as inside the
    # fused step: each kernel launched back to back as a programmatic
    # dependent of the one before (tts_set_launch_flags), over inputs larger
    # than L2 so that no launch finds its bytes cached: attention alternates
    # two copies of the cache, tables and queries; the head rotates 16 copies
    # of W.  One pair of events around each run; mean per launch.
    gpu_out = step.out.detach().cpu()
    gpu_ids = step.ids.detach().cpu().numpy()
    att_us_iso = 1e3 * statistics.fmean(t_att)
    head_us_iso = 1e3 * statistics.fmean(t_head)
    cache2 = bd.KVCache(cache.k_pool.clone(), cache.v_pool.clone()) if args.chained else None
    d2 = {k: d[k].clone() for k in ("block_table", "ctx_lens", "q")}
    attn_sets = [(cache, d["block_table"], d["ctx_lens"], d["q"], step.attn_ws),
                 (cache2, d2["block_table"], d2["ctx_lens"], d2["q"], torch.zeros_like(step.attn_ws))]
    out2 = torch.empty_like(step.out)
    W_copies = [W] + ([W.clone() for _ in range(15)] if args.chained else [])
    # launches per captured chain: a multiple of the two attention input sets
    # and of the 16 copies of W; the chain is replayed n_rep times
    n_graph = 32
    n_rep = max(2, -(-min(K, 400) // n_graph))

    def chained(fn):
        """Mean per-launch time of fn(0), fn(1), ... captured once as a CUDA
        graph with each launch a programmatic dependent of the one before,
        the graph replayed n_rep times between two events.  Capturing keeps
        the binding's host cost per call (about 13 us for the attention, 20 us
        for the head) out of the chain, which a host loop would make the
        bottleneck for kernels shorter than that."""
        for i in range(4):
            fn(i)
        torch.cuda.synchronize()
        prev = bd.tts_set_launch_flags(bd._lib.LAUNCH_PROGRAMMATIC)
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                for i in range(n_graph):
                    fn(i)
        finally:
            bd.tts_set_launch_flags(prev)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_rep):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        del g
        return e0.elapsed_time(e1) * 1e3 / (n_rep * n_graph)

    def attn_i(i):
        c, tbl, lens, q, ws = attn_sets[i & 1]
        bd.tts_decode_attn(c, tbl, lens, w.ctx_hi, q, step.out if i & 1 == 0 else out2, ws, step.scale, w.causal,
                           err=step.err)

    def head_i(i):
        bd.tts_codebook_head_select(step.out.view(step.R, -1), W_copies[i % len(W_copies)], step.ids, step.head_ws,
                                    mode=mode, temperature=w.T, seed=seed, step=stp)

    if args.chained:
        att_chain_us = chained(attn_i)
        head_chain_us = chained(head_i)
    else:
        att_chain_us, head_chain_us = att_us_iso, head_us_iso
    del cache2, d2, out2, W_copies, attn_sets
    torch.cuda.empty_cache()

    # ---- end to end through the public API with host buffers: the library's
    # captured step copies the step's inputs in from pinned host memory, runs
    # the step and writes the ids back; wall clock, synchronised every step.
    from decode_step_gb300.step import GraphedStep
    g_inputs = {k: d[k] for k in names}
    if mode == bd.TTS_GUMBEL:
        g_inputs["seed"], g_inputs["step"] = seed, stp
    graphed = GraphedStep(step, g_inputs)
    h2d = graphed.h2d_bytes
    d2h = step.R * 4
    n_e2e = max(10, min(args.e2e_steps, K))
    for _ in range(5):
        graphed()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        graphed()
    e2e_s = time.perf_counter() - t0
    e2e_all = max_over_ranks(e2e_s / n_e2e * 1e3, world, device)
    _, e2e_value = combine_rank_times(e2e_all, w.B * w.q_len)

    # ---- the captured-step set: graphs for batch sizes 1, 2, 4, ..., B; a
    # step with n active streams runs the smallest size >= n (the rest padded
    # onto a spare block); wall clock per step, host writes included.
    e2e_sizes = {}
    sizes_req = [int(x) for x in args.e2e_sizes.split(",") if x.strip()] if rank == 0 else []
    if sizes_req:
        from decode_step_gb300.step import GraphedStepSet
        used = set(int(x) for x in inp["block_table"][inp["block_table"] >= 0].ravel())
        spare = sorted(set(range(inp["num_blocks"])) - used)
        sizes = [s for s in (1, 2, 4, 8, 16, 32, 64, 128, 256) if s < w.B] + [w.B]
        if spare:
            gset = GraphedStepSet(step, g_inputs, sizes, scratch_block=spare[0])
            host_arrays = {k: t.detach().cpu() for k, t in g_inputs.items()}
            for n in sizes_req:
                if not 1 <= n <= w.B:
                    continue
                # the n streams' inputs written into the pinned views once (as
                # the single-graph e2e above); each step: launch, sync, read ids
                gset.step_streams({k: t[:n] for k, t in host_arrays.items()})
                for _ in range(5):
                    gset.launch(n)
                reps = max(20, n_e2e // 4)
                t0 = time.perf_counter()
                for _ in range(reps):
                    gset.launch(n)
                us = (time.perf_counter() - t0) / reps * 1e6
                e2e_sizes[str(n)] = {"us_per_step": us, "tokens_per_s": n * w.q_len / (us * 1e-6),
                                     "graph_size": next(s for s in sizes if s >= n)}
            del gset

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    peaks, peak_kind = load_peaks()
    att_us = 1e3 * statistics.fmean(t_att)
    head_us = 1e3 * statistics.fmean(t_head)
    app_us = 1e3 * statistics.fmean(t_app)
    ab = attn_bytes(inp)
    achieved = ab / (att_chain_us * 1e-6) / 1e9
    hb = head_bytes(w)
    head_gbs = hb / (head_chain_us * 1e-6) / 1e9
    head_tflops = 2.0 * w.R * w.H * w.V / (head_chain_us * 1e-6) / 1e12
    traffic = recorded_traffic("decode_attn", w.name)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "impl": "native",
        "config": workload_config(w, world),
        "roofline": {"bound": "hbm", "kernel": "decode_attn", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": traffic, "algorithmic_bytes": ab, "launch_us": att_chain_us,
                     "timing": (f"{n_graph} launches captured as one CUDA graph, each a programmatic dependent "
                                f"of the one before, alternating two copies of the inputs (2 x cache > L2); the "
                                f"graph replayed {n_rep} times between CUDA events")
                     if args.chained else "single launches after an L2 flush (chained pass skipped)",
                     "achieved_isolated": ab / (att_us * 1e-6) / 1e9,
                     "frac_isolated": ab / (att_us * 1e-6) / 1e9 / peaks["hbm_gbs"],
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback"},
        "kernels": {
            "decode_attn_us_chained": att_chain_us, "head_select_us_chained": head_chain_us,
            "chained_note": "per-kernel time with the launch latency hidden (a captured chain of launches, "
                            "each a programmatic dependent of the one before, inputs rotated beyond L2); the "
                            "*_us keys below are "
                            "single launches after an L2 flush, each bracketed by events (launch latency "
                            "included)",
            "kv_append_us": app_us, "decode_attn_us": att_us, "head_select_us": head_us,
            "step_us": 1e3 * ms,
            "sum_of_kernels_us": app_us + att_us + head_us,
            "decode_attn_us_median": 1e3 * statistics.median(t_att),
            "head_select_us_median": 1e3 * statistics.median(t_head),
            "kv_append_gbs": append_bytes(w) / (app_us * 1e-6) / 1e9,
            "write_only_flush": {"decode_attn_us": 1e3 * statistics.fmean(t_att_w),
                                 "head_select_us": 1e3 * statistics.fmean(t_head_w),
                                 "launches": K3},
            "head_roofline": {"bound": "hbm", "achieved": head_gbs, "peak": peaks["hbm_gbs"],
                              "unit": "GB/s", "frac": head_gbs / peaks["hbm_gbs"],
                              "algorithmic_bytes": hb, "tflops": head_tflops, "launch_us": head_chain_us,
                              "frac_isolated": hb / (head_us * 1e-6) / 1e9 / peaks["hbm_gbs"]},
        },
        "gpu_launches": 3 * K,
        "step_note": "each timed step is one tts_decode_step call (append, attention, head; "
                     "the last two launched as programmatic dependents); per-kernel times come "
                     "from a separate pass launching the kernels one by one",
        "device_error_flags": errflags,
        "clocks": clk,
        # context: a voice at 12.5 frames/s over 4 retained codebook streams
        # consumes 50 codec tokens/s per layer-step
        "realtime_voice_equivalents": value / (12.5 * 4),
        "e2e_by_active_streams": e2e_sizes,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": n_e2e, "note": "wall clock; tts_step_graph (one CUDA graph captured by the "
                                        "library): every input of the step crosses from pinned host "
                                        "memory each step (the append and the attention's tile map read "
                                        "theirs there directly, a copy kernel moves the query rows to the "
                                        "device), the step runs, the ids and a boundary-token count are "
                                        "written to pinned host memory; the host calls tts_step_graph_run "
                                        "(launch, then wait for the ids) every step"},
    }
    if world == 1:
        g_out = wl.to_f32(gpu_out.view(torch.int16).numpy().view(np.uint16), w.dtype) if w.dtype == "bf16" \
            else gpu_out.numpy()
        line["cpu_baseline"], line["parity"] = cpu_baseline(inp, args.cpu_seconds, g_out.astype(np.float64), gpu_ids)
        ids = [x.strip() for x in args.sweep.split(",") if x.strip()]
        if ids:
            del step, graphed, cache, W, d
            torch.cuda.empty_cache()
            line["workloads"] = kernel_sweep(ids, args.sweep_reps, flush_l2, peaks, device)
        if args.code_predictor:
            line["code_predictor"] = predictor_sweep(args.sweep_reps, flush_l2, peaks, device)
        heads = [x.strip() for x in args.audio_heads.split(",") if x.strip()]
        if heads:
            line["audio_heads"] = audio_head_sweep(heads, args.sweep_reps, flush_l2, peaks, device)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
