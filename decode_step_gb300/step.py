"""One batched decode step through the C ABI: append, attend, score and pick.

`DecodeStep` owns the workspaces and output buffers for a fixed batch shape
and issues tts_decode_step (append -> attention -> head, the later kernels
launched as programmatic dependents) on one stream.  The attention output
[B][q_len][Hq][D] is read by the head as h [B * q_len][Hq * D], so Hq * D must
equal the head's hidden width.

`GraphedStep` wraps tts_step_graph: a whole serving step captured once by the
library for fixed buffers (the copy of the step's inputs from pinned host
memory, the decode step, the chosen ids and a boundary-token count back to
pinned host memory).  Each step then is: write the pinned inputs, launch,
synchronise, read the pinned ids.
"""
from __future__ import annotations

import math

import torch

from . import binding as bd


class DecodeStep:
    def __init__(self, cache: bd.KVCache, W: torch.Tensor, num_q_heads: int, B: int,
                 max_ctx_len: int, q_len: int = 1, causal: bool = False,
                 mode: int = bd.TTS_ARGMAX, temperature: float = 0.0, scale: float | None = None,
                 rope_base: float = 0.0):
        dev = cache.k_pool.device
        self.cache, self.W = cache, W
        self.B, self.q_len, self.Hq = B, q_len, num_q_heads
        self.max_ctx_len, self.causal = max_ctx_len, causal
        self.mode, self.temperature = mode, temperature
        self.rope_base = rope_base  # != 0: q and k_new rotated at their positions (q in place)
        self.scale = 1.0 / math.sqrt(cache.head_dim) if scale is None else scale
        H = num_q_heads * cache.head_dim
        if W.shape[1] != H:
            raise ValueError(f"head width {W.shape[1]} != num_q_heads * head_dim = {H}")
        self.R, self.V = B * q_len, W.shape[0]
        attn_ws = bd.tts_decode_attn_workspace_size(B, q_len, num_q_heads, cache.num_kv_heads,
                                                    cache.head_dim, max_ctx_len)
        head_ws = bd.tts_head_workspace_size(self.R, self.V)
        if attn_ws == 0 or head_ws == 0:
            raise ValueError("unsupported decode-step shape")
        self.attn_ws = torch.zeros(attn_ws, dtype=torch.uint8, device=dev)
        self.head_ws = torch.zeros(head_ws, dtype=torch.uint8, device=dev)
        self.out = torch.empty((B, q_len, num_q_heads, cache.head_dim), dtype=cache.dtype, device=dev)
        self.ids = torch.empty(self.R, dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def __call__(self, block_table, ctx_before, ctx_lens, q, k_new, v_new, seed=None, step=None,
                 eos_allowed=None, logits_out=None, best=None, stream=None) -> torch.Tensor:
        """Runs the step; returns the device tensor of chosen ids [B * q_len]."""
        bd.tts_decode_step(self.cache, block_table, ctx_before, ctx_lens, self.max_ctx_len, q, k_new,
                           v_new, self.out, self.attn_ws, self.scale, self.W, self.ids, self.head_ws,
                           causal=self.causal, mode=self.mode, temperature=self.temperature,
                           seed=seed, step=step, eos_allowed=eos_allowed, best=best,
                           logits_out=logits_out, err=self.err, stream=stream, rope_base=self.rope_base)
        return self.ids


class GraphedStep:
    """A captured serving step: pinned host inputs -> device -> step -> pinned ids.

    `inputs` maps names of DecodeStep's call arguments (block_table, ctx_before,
    ctx_lens, q, k_new, v_new, and optionally seed, step) to tensors giving
    each input's shape, dtype and first contents.  The step's inputs live in
    one pinned host buffer mirrored by one device buffer (`host[name]` and
    `dev[name]` are views into them, 256-byte aligned).  The library captures
    the whole step once (tts_step_graph_create): a launch copies the packed
    inputs with one kernel reading the pinned buffer, runs the step, and writes
    the ids and the count of rows that picked the boundary token into pinned
    host memory.  Write a step's inputs into `host[...]`, call the object, read
    the ids it returns (`boundary_count` holds the count).  With draft_probs,
    draft_tokens, vseed and vstep among the inputs (a q_len = K + 1 step) the
    captured step also verifies the drafts against the head's logits;
    `n_accepted_host` / `next_token_host` then hold the result.
    """

    NAMES = ("block_table", "ctx_before", "ctx_lens", "q", "k_new", "v_new", "seed", "step",
             "draft_probs", "draft_tokens", "vseed", "vstep")

    def __init__(self, step: DecodeStep, inputs: dict, stream: torch.cuda.Stream | None = None,
                 verify_temperature: float | None = None, bonus: bool = False):
        self.step = step
        offsets, total = {}, 0
        for k, t in inputs.items():
            if k not in self.NAMES:
                raise ValueError(f"unknown step input {k}")
            offsets[k] = total
            total += -(-(t.numel() * t.element_size()) // 256) * 256
        device = next(iter(inputs.values())).device
        self.host_blob = torch.empty(total, dtype=torch.uint8, device="cpu").pin_memory()
        self.dev_blob = torch.empty(total, dtype=torch.uint8, device=device)
        self.host, self.dev = {}, {}
        for k, t in inputs.items():
            n = t.numel() * t.element_size()
            self.host[k] = self.host_blob[offsets[k]:offsets[k] + n].view(t.dtype).view(t.shape)
            self.dev[k] = self.dev_blob[offsets[k]:offsets[k] + n].view(t.dtype).view(t.shape)
            self.host[k].copy_(t.detach().cpu())
        self.ids_host = torch.zeros(step.R, dtype=torch.int32, device="cpu").pin_memory()
        self.boundary_host = torch.zeros(1, dtype=torch.int32, device="cpu").pin_memory()
        self.stream = torch.cuda.Stream() if stream is None else stream
        d = self.dev
        # speculative verify inside the captured step: the head keeps its
        # logits for the K + 1 rows of every stream and verify reads them
        verify, self.logits = None, None
        self.n_accepted_host = self.next_token_host = None
        if "draft_probs" in inputs:
            B = step.B
            self.logits = torch.empty((step.R, step.V), dtype=torch.float32, device=device)
            self.n_accepted_host = torch.zeros(B, dtype=torch.int32, device="cpu").pin_memory()
            self.next_token_host = torch.zeros(B, dtype=torch.int32, device="cpu").pin_memory()
            verify = dict(draft_probs=d["draft_probs"], draft_tokens=d["draft_tokens"],
                          temperature=verify_temperature, bonus=bonus, vseed=d["vseed"], vstep=d["vstep"],
                          n_accepted=torch.empty(B, dtype=torch.int32, device=device),
                          next_token=torch.empty(B, dtype=torch.int32, device=device),
                          h_n_accepted=self.n_accepted_host, h_next_token=self.next_token_host)
        self.graph = bd.StepGraph(
            step.cache, d["block_table"], d["ctx_before"], d["ctx_lens"], step.max_ctx_len, d["q"],
            d["k_new"], d["v_new"], step.out, step.attn_ws, step.scale, step.W, step.ids, step.head_ws,
            self.host_blob, self.dev_blob, self.ids_host, self.boundary_host, causal=step.causal,
            mode=step.mode, temperature=step.temperature, seed=d.get("seed"), step=d.get("step"),
            err=step.err, rope_base=step.rope_base, logits_out=self.logits, verify=verify)

    @property
    def h2d_bytes(self) -> int:
        """Bytes a launch copies from the pinned input buffer (inputs and padding)."""
        return self.host_blob.numel()

    @property
    def boundary_count(self) -> int:
        """Rows whose id is the boundary token in the last completed launch."""
        return int(self.boundary_host.item())

    def __call__(self) -> torch.Tensor:
        """Runs the captured step and returns the (pinned, host) ids once they
        are there (tts_step_graph_run: a spin on the launch number the head
        writes after them, or a stream synchronisation)."""
        self.graph.run(self.stream)
        return self.ids_host


def choose_size(sizes, n: int):
    """The smallest captured size that holds n streams, or None."""
    for s in sizes:
        if s >= n:
            return s
    return None


def cohorts(n: int, largest: int):
    """Split n streams into consecutive cohorts of at most `largest`: (first, count)."""
    return [(s, min(largest, n - s)) for s in range(0, n, largest)]


class GraphedStepSet:
    """Captured serving steps for a set of batch sizes (tts_step_graph_set).

    `step` is a DecodeStep for the largest size B; `inputs` maps input names
    (as GraphedStep) to tensors with B streams in their first dimension.  One
    pinned host buffer and its device mirror hold every input, one region per
    name laid out for B streams; the graph of size b copies the first b rows
    of each region.  `scratch_block` is a KV block no stream uses: streams past
    the active ones of a launch get a table row of it, one new token at
    position 0 and zero rows, so their work is harmless; their ids are
    dropped.  `step_streams(arrays)` runs any number of streams: each cohort of
    at most B streams is copied into the first rows, padded to the smallest
    captured size, launched and read back.
    """

    PAD = {"ctx_before": 0, "q": 0, "k_new": 0, "v_new": 0, "seed": 0, "step": 0}

    def __init__(self, step: DecodeStep, inputs: dict, sizes, scratch_block: int,
                 stream: torch.cuda.Stream | None = None):
        self.step, self.B = step, step.B
        self.sizes = sorted(int(s) for s in sizes)
        if self.sizes[-1] != self.B:
            raise ValueError("the largest size must be the DecodeStep's batch")
        offsets, total, rows = {}, 0, {}
        for k, t in inputs.items():
            if k not in GraphedStep.NAMES:
                raise ValueError(f"unknown step input {k}")
            if t.shape[0] != self.B:
                raise ValueError(f"{k} must hold {self.B} streams in its first dimension")
            offsets[k] = total
            rows[k] = t.numel() * t.element_size() // self.B
            total += -(-(t.numel() * t.element_size()) // 256) * 256
        device = next(iter(inputs.values())).device
        self.host_blob = torch.empty(total, dtype=torch.uint8, device="cpu").pin_memory()
        self.dev_blob = torch.empty(total, dtype=torch.uint8, device=device)
        self.host, self.dev = {}, {}
        for k, t in inputs.items():
            n = t.numel() * t.element_size()
            self.host[k] = self.host_blob[offsets[k]:offsets[k] + n].view(t.dtype).view(t.shape)
            self.dev[k] = self.dev_blob[offsets[k]:offsets[k] + n].view(t.dtype).view(t.shape)
            self.host[k].copy_(t.detach().cpu())
        self.regions = [(offsets[k], rows[k]) for k in inputs]
        self.scratch_block = int(scratch_block)
        self.ids_host = torch.zeros(step.R, dtype=torch.int32, device="cpu").pin_memory()
        self.boundary_host = torch.zeros(1, dtype=torch.int32, device="cpu").pin_memory()
        self.stream = torch.cuda.Stream() if stream is None else stream
        d = self.dev
        self.graphs = bd.StepGraphSet(
            step.cache, d["block_table"], d["ctx_before"], d["ctx_lens"], step.max_ctx_len, d["q"],
            d["k_new"], d["v_new"], step.out, step.attn_ws, step.scale, step.W, step.ids, step.head_ws,
            self.host_blob, self.dev_blob, self.ids_host, self.sizes, self.regions, self.boundary_host,
            causal=step.causal, mode=step.mode, temperature=step.temperature, seed=d.get("seed"),
            step=d.get("step"), err=step.err, rope_base=step.rope_base)

    def _pad(self, n: int, b: int) -> None:
        """Streams n..b-1: the scratch block, one new token at position 0, zero rows."""
        if b <= n:
            return
        h = self.host
        h["block_table"][n:b] = self.scratch_block
        h["ctx_lens"][n:b] = self.step.q_len
        for k, v in self.PAD.items():
            if k in h:
                h[k][n:b] = v

    def launch(self, n: int) -> torch.Tensor:
        """Runs the first n streams as currently written in `host` (n at most
        the largest size); returns the pinned ids of those streams."""
        b = choose_size(self.sizes, n)
        if b is None:
            raise ValueError(f"{n} streams exceed the largest captured size {self.sizes[-1]}")
        self._pad(n, b)
        chosen = self.graphs.run(n, self.stream)
        assert chosen == b
        return self.ids_host[:n * self.step.q_len]

    def step_streams(self, arrays: dict) -> torch.Tensor:
        """One decode step for every stream of `arrays` (host tensors keyed
        like `inputs`, streams in the first dimension, any count): cohorts of
        at most the largest size run one after another.  Returns the ids."""
        n = next(iter(arrays.values())).shape[0]
        out = []
        for first, count in cohorts(n, self.B):
            for k, t in arrays.items():
                self.host[k][:count] = t[first:first + count]
            out.append(self.launch(count).clone())
        return torch.cat(out) if out else torch.empty(0, dtype=torch.int32)
