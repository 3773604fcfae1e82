"""Python binding of the C ABI (include/tts_decode.h), same function names.

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the computation runs in the library's kernels.
Shapes and dtypes are checked here so a mistake raises a Python error before
anything is launched.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (TTS_ARGMAX, TTS_BF16, TTS_F32, TTS_FP8_E4M3, TTS_GUMBEL, TTS_VERIFY_BONUS,  # noqa: F401
                   KVCacheDesc, TTSError, check, lib)

_DTYPES = {torch.float32: TTS_F32, torch.bfloat16: TTS_BF16}


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return _ptr(t)


def _keys(t: torch.Tensor | None, name: str, n: int):
    """uint64 (or same-width int64) key arrays."""
    if t is None:
        return None
    if t.dtype not in (torch.uint64, torch.int64):
        raise ValueError(f"{name} must be uint64 (or int64 with the same bits)")
    return _dev(t, name, None, (n,))


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class KVCache:
    """Paged KV pool.

    float32 / bfloat16: k_pool, v_pool [num_blocks][num_kv_heads][16][head_dim].
    FP8 E4M3: k_pool uint8 [num_blocks][num_kv_heads][4224], one record per
    (block, KV head) in the layout of tts_kv_cache (key codes, value codes,
    key and value scales), v_pool None; head_dim is 128 and the step's
    activations are bfloat16.
    """

    FP8_TILE_BYTES = 4224

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor | None = None):
        self.fp8 = k_pool.dtype == torch.uint8
        if self.fp8:
            if v_pool is not None or k_pool.dim() != 3 or k_pool.shape[2] != self.FP8_TILE_BYTES:
                raise ValueError("an FP8 cache is one uint8 tensor [num_blocks][num_kv_heads][4224]")
            nb, hkv, _ = k_pool.shape
            d = 128
            dtype = TTS_FP8_E4M3
            vptr = None
        else:
            if v_pool is None or k_pool.shape != v_pool.shape or k_pool.dim() != 4 or k_pool.shape[2] != 16:
                raise ValueError("pools must be [num_blocks][num_kv_heads][16][head_dim] and alike")
            if k_pool.dtype != v_pool.dtype or k_pool.dtype not in _DTYPES:
                raise ValueError("pools must both be float32 or bfloat16 (or an FP8 uint8 tile array)")
            nb, hkv, _, d = k_pool.shape
            dtype = _DTYPES[k_pool.dtype]
            vptr = _dev(v_pool, "v_pool")
        self.k_pool, self.v_pool = k_pool, v_pool
        self.desc = KVCacheDesc(nb, 16, hkv, d, dtype, _dev(k_pool, "k_pool"), vptr)

    @property
    def num_blocks(self) -> int:
        return self.desc.num_blocks

    @property
    def num_kv_heads(self) -> int:
        return self.desc.num_kv_heads

    @property
    def head_dim(self) -> int:
        return self.desc.head_dim

    @property
    def dtype(self) -> torch.dtype:
        """Element type of the step's activations (q, k_new, v_new, attention output)."""
        return torch.bfloat16 if self.fp8 else self.k_pool.dtype


class BlockPool:
    """Host free list of KV block ids (tts_block_pool_*)."""

    def __init__(self, num_blocks: int):
        h = ctypes.c_void_p()
        check("tts_block_pool_create", lib().tts_block_pool_create(num_blocks, ctypes.byref(h)))
        self._h = h

    def alloc(self, n: int) -> list[int]:
        ids = (ctypes.c_int32 * max(n, 1))()
        check("tts_block_pool_alloc", lib().tts_block_pool_alloc(self._h, n, ids))
        return list(ids[:n])

    def free(self, ids) -> None:
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        check("tts_block_pool_free", lib().tts_block_pool_free(self._h, arr, len(ids)))

    @property
    def num_free(self) -> int:
        n = lib().tts_block_pool_num_free(self._h)
        if n < 0:
            check("tts_block_pool_num_free", n)
        return n

    def close(self) -> None:
        if self._h:
            lib().tts_block_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tts_kv_append(cache: KVCache, block_table, ctx_before, k_new, v_new, err=None, stream=None):
    B, max_blocks = block_table.shape
    q_len = k_new.shape[1]
    shape = (B, q_len, cache.num_kv_heads, cache.head_dim)
    args = (ctypes.byref(cache.desc), _dev(block_table, "block_table", torch.int32), max_blocks,
            _dev(ctx_before, "ctx_before", torch.int32, (B,)), B, q_len,
            _dev(k_new, "k_new", cache.dtype, shape), _dev(v_new, "v_new", cache.dtype, shape),
            None if err is None else _dev(err, "err", torch.int32), _stream(stream))
    check("tts_kv_append", lib().tts_kv_append(*args))


def tts_kv_append_rope(cache: KVCache, block_table, ctx_before, q, k_new, v_new, rope_base=10000.0,
                       err=None, stream=None):
    """tts_kv_append with the rotary embedding of q (in place) and k_new at
    positions ctx_before[b] + j; q is [B][q_len][Hq][head_dim] bf16."""
    B, max_blocks = block_table.shape
    q_len, Hq = k_new.shape[1], q.shape[2]
    shape = (B, q_len, cache.num_kv_heads, cache.head_dim)
    args = (ctypes.byref(cache.desc), _dev(block_table, "block_table", torch.int32), max_blocks,
            _dev(ctx_before, "ctx_before", torch.int32, (B,)), B, q_len, Hq, float(rope_base),
            _dev(q, "q", cache.dtype, (B, q_len, Hq, cache.head_dim)),
            _dev(k_new, "k_new", cache.dtype, shape), _dev(v_new, "v_new", cache.dtype, shape),
            None if err is None else _dev(err, "err", torch.int32), _stream(stream))
    check("tts_kv_append_rope", lib().tts_kv_append_rope(*args))


def tts_decode_attn_workspace_size(B, q_len, num_q_heads, num_kv_heads, head_dim, max_ctx_len) -> int:
    return int(lib().tts_decode_attn_workspace_size(B, q_len, num_q_heads, num_kv_heads, head_dim,
                                                   max_ctx_len))


def tts_decode_attn(cache: KVCache, block_table, ctx_lens, max_ctx_len, q, out, ws, scale,
                    causal=False, err=None, stream=None):
    B, max_blocks = block_table.shape
    _, q_len, Hq, D = q.shape
    args = (ctypes.byref(cache.desc), _dev(block_table, "block_table", torch.int32), max_blocks,
            _dev(ctx_lens, "ctx_lens", torch.int32, (B,)), int(max_ctx_len), B, q_len, Hq,
            float(scale), int(bool(causal)), _dev(q, "q", cache.dtype, (B, q_len, Hq, cache.head_dim)),
            _dev(out, "out", cache.dtype, (B, q_len, Hq, cache.head_dim)), _dev(ws, "ws"),
            ws.numel() * ws.element_size(), None if err is None else _dev(err, "err", torch.int32),
            _stream(stream))
    check("tts_decode_attn", lib().tts_decode_attn(*args))


def tts_decode_attn_noalloc(cache: KVCache, block_table, ctx_lens, max_ctx_len, q, out, scale,
                            causal=False, err=None, stream=None):
    """tts_decode_attn without a workspace, for callers that cannot allocate
    device memory where they run a step (all free memory given to the KV
    pool, a host without an allocator, a frame budget that cannot absorb
    cudaMalloc's synchronisation); uses the library's 16 MiB static scratch,
    shared by all calls."""
    B, max_blocks = block_table.shape
    _, q_len, Hq, D = q.shape
    args = (ctypes.byref(cache.desc), _dev(block_table, "block_table", torch.int32), max_blocks,
            _dev(ctx_lens, "ctx_lens", torch.int32, (B,)), int(max_ctx_len), B, q_len, Hq,
            float(scale), int(bool(causal)), _dev(q, "q", cache.dtype, (B, q_len, Hq, cache.head_dim)),
            _dev(out, "out", cache.dtype, (B, q_len, Hq, cache.head_dim)),
            None if err is None else _dev(err, "err", torch.int32), _stream(stream))
    check("tts_decode_attn_noalloc", lib().tts_decode_attn_noalloc(*args))


def tts_head_workspace_size(R, V) -> int:
    return int(lib().tts_head_workspace_size(R, V))


def tts_codebook_head_select(h, W, ids, ws, mode=TTS_ARGMAX, temperature=0.0, seed=None, step=None,
                             eos_allowed=None, best=None, logits_out=None, stream=None):
    R, H = h.shape
    V = W.shape[0]
    if h.dtype not in _DTYPES or W.dtype != h.dtype or W.shape[1] != H:
        raise ValueError("h [R][H] and W [V][H] must share a float32 / bfloat16 dtype")
    args = (_dev(h, "h"), _dev(W, "W"), _DTYPES[h.dtype], R, H, V, int(mode), float(temperature),
            _keys(seed, "seed", R), _keys(step, "step", R),
            None if eos_allowed is None else _dev(eos_allowed, "eos_allowed", torch.uint8, (R,)),
            _dev(ids, "ids", torch.int32, (R,)),
            None if best is None else _dev(best, "best", torch.float32, (R,)),
            None if logits_out is None else _dev(logits_out, "logits_out", torch.float32, (R, V)),
            _dev(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    check("tts_codebook_head_select", lib().tts_codebook_head_select(*args))


def tts_audio_head_select(h, W1, b1, W2, b2, z, ids, ws, mode=TTS_ARGMAX, temperature=0.0, seed=None, step=None,
                          n_tail=0, tail_allowed=None, best=None, logits_out=None, stream=None):
    """The two-layer audio head: z = bf16(Mish(h W1^T + b1)) written to `z`
    [R][F], then the head over z W2^T + b2 with the last n_tail ids masked per
    row by tail_allowed (uint32 bits; None: all allowed).  bf16 weights; b1 / b2
    float32 or None."""
    R, H = h.shape
    F, V = W1.shape[0], W2.shape[0]
    for t, n in ((h, "h"), (W1, "W1"), (W2, "W2"), (z, "z")):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{n} must be bfloat16")
    if W1.shape[1] != H or W2.shape[1] != F:
        raise ValueError("W1 must be [F][H] and W2 [V][F]")
    args = (_dev(h, "h"), _dev(W1, "W1"), None if b1 is None else _dev(b1, "b1", torch.float32, (F,)),
            _dev(W2, "W2"), None if b2 is None else _dev(b2, "b2", torch.float32, (V,)), R, H, F, V, int(n_tail),
            None if tail_allowed is None else _dev(tail_allowed, "tail_allowed", torch.int32, (R,)),
            int(mode), float(temperature), _keys(seed, "seed", R), _keys(step, "step", R),
            _dev(z, "z", torch.bfloat16, (R, F)), _dev(ids, "ids", torch.int32, (R,)),
            None if best is None else _dev(best, "best", torch.float32, (R,)),
            None if logits_out is None else _dev(logits_out, "logits_out", torch.float32, (R, V)),
            _dev(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    check("tts_audio_head_select", lib().tts_audio_head_select(*args))


def tts_spec_verify(target_logits, draft_probs, draft_tokens, temperature, seed, step,
                    n_accepted, next_token, bonus=False, err=None, stream=None):
    B, K1, V = target_logits.shape
    K = K1 - 1
    args = (_dev(target_logits, "target_logits", torch.float32),
            _dev(draft_probs, "draft_probs", torch.float32, (B, K, V)),
            _dev(draft_tokens, "draft_tokens", torch.int32, (B, K)), B, K, V, float(temperature),
            _keys(seed, "seed", B), _keys(step, "step", B),
            TTS_VERIFY_BONUS if bonus else 0, _dev(n_accepted, "n_accepted", torch.int32, (B,)),
            _dev(next_token, "next_token", torch.int32, (B,)),
            None if err is None else _dev(err, "err", torch.int32), _stream(stream))
    check("tts_spec_verify", lib().tts_spec_verify(*args))


def _step_args(cache: KVCache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new,
               attn_out, attn_ws, scale, W, ids, head_ws, causal, rope_base, mode, temperature, seed, step,
               eos_allowed, best, logits_out, err, stream):
    """tts_decode_step's argument tuple (the cache as a byref, the stream last)."""
    B, max_blocks = block_table.shape
    _, q_len, Hq, D = q.shape
    kv_shape = (B, q_len, cache.num_kv_heads, cache.head_dim)
    R, V = B * q_len, W.shape[0]
    if W.dtype != cache.dtype or W.shape[1] != Hq * D:
        raise ValueError("W must be [V][num_q_heads * head_dim] in the cache dtype")
    args = (ctypes.byref(cache.desc), _dev(block_table, "block_table", torch.int32), max_blocks,
            _dev(ctx_before, "ctx_before", torch.int32, (B,)), _dev(ctx_lens, "ctx_lens", torch.int32, (B,)),
            int(max_ctx_len), B, q_len, Hq, float(scale), int(bool(causal)), float(rope_base),
            _dev(q, "q", cache.dtype, (B, q_len, Hq, cache.head_dim)),
            _dev(k_new, "k_new", cache.dtype, kv_shape), _dev(v_new, "v_new", cache.dtype, kv_shape),
            _dev(attn_out, "attn_out", cache.dtype, (B, q_len, Hq, cache.head_dim)), _dev(attn_ws, "attn_ws"),
            attn_ws.numel() * attn_ws.element_size(), _dev(W, "W"), V, int(mode), float(temperature),
            _keys(seed, "seed", R), _keys(step, "step", R),
            None if eos_allowed is None else _dev(eos_allowed, "eos_allowed", torch.uint8, (R,)),
            _dev(ids, "ids", torch.int32, (R,)),
            None if best is None else _dev(best, "best", torch.float32, (R,)),
            None if logits_out is None else _dev(logits_out, "logits_out", torch.float32, (R, V)),
            _dev(head_ws, "head_ws"), head_ws.numel() * head_ws.element_size(),
            None if err is None else _dev(err, "err", torch.int32), _stream(stream))
    return args


def tts_decode_step(cache: KVCache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new,
                    attn_out, attn_ws, scale, W, ids, head_ws, causal=False, mode=TTS_ARGMAX,
                    temperature=0.0, seed=None, step=None, eos_allowed=None, best=None,
                    logits_out=None, err=None, stream=None, rope_base=0.0):
    """rope_base != 0 rotates q (in place) and k_new at positions ctx_before[b] + j."""
    args = _step_args(cache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new, attn_out,
                      attn_ws, scale, W, ids, head_ws, causal, rope_base, mode, temperature, seed, step,
                      eos_allowed, best, logits_out, err, stream)
    check("tts_decode_step", lib().tts_decode_step(*args))


def _pinned(t: torch.Tensor, name: str, dtype=None, numel=None):
    if t.is_cuda or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements")
    return ctypes.c_void_p(t.data_ptr())


def _graph_desc(cache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new, attn_out, attn_ws, scale,
                W, ids, head_ws, h_inputs, d_inputs, h_ids, h_boundary_count, causal, mode, temperature, seed, step,
                eos_allowed, best, logits_out, err, rope_base, verify=None):
    args = _step_args(cache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new, attn_out,
                      attn_ws, scale, W, ids, head_ws, causal, rope_base, mode, temperature, seed, step,
                      eos_allowed, best, logits_out, err, None)
    R = ids.numel()
    nbytes = h_inputs.numel() * h_inputs.element_size()
    if d_inputs.numel() * d_inputs.element_size() != nbytes or not d_inputs.is_cuda:
        raise ValueError("d_inputs must be a device tensor of h_inputs' size")
    host = (_pinned(h_inputs, "h_inputs"), _dev(d_inputs, "d_inputs"), nbytes,
            _pinned(h_ids, "h_ids", torch.int32, R),
            None if h_boundary_count is None else _pinned(h_boundary_count, "h_boundary_count", torch.int32, 1))
    desc = _lib.StepGraphDesc(ctypes.pointer(cache.desc), *args[1:-1], *host)
    if verify is not None:
        B = block_table.shape[0]
        K = q.shape[1] - 1
        V = W.shape[0]
        v = verify
        desc.d_draft_probs = _dev(v["draft_probs"], "draft_probs", torch.float32, (B, K, V))
        desc.d_draft_tokens = _dev(v["draft_tokens"], "draft_tokens", torch.int32, (B, K))
        desc.verify_temperature = float(v["temperature"])
        desc.verify_flags = TTS_VERIFY_BONUS if v.get("bonus") else 0
        desc.d_vseed = _keys(v["vseed"], "vseed", B)
        desc.d_vstep = _keys(v["vstep"], "vstep", B)
        desc.d_n_accepted = _dev(v["n_accepted"], "n_accepted", torch.int32, (B,))
        desc.d_next_token = _dev(v["next_token"], "next_token", torch.int32, (B,))
        if v.get("h_n_accepted") is not None:
            desc.h_n_accepted = _pinned(v["h_n_accepted"], "h_n_accepted", torch.int32, B)
        if v.get("h_next_token") is not None:
            desc.h_next_token = _pinned(v["h_next_token"], "h_next_token", torch.int32, B)
    return desc


class StepGraph:
    """tts_step_graph_*: a decode step captured once as a CUDA graph.

    Takes tts_decode_step's arguments (its input tensors normally views into
    `d_inputs`) plus the host side: `h_inputs` (pinned, copied to `d_inputs`
    by every launch), `h_ids` (pinned int32 [B * q_len], written by every
    launch) and optionally `h_boundary_count` (pinned int32 [1]: rows whose id
    is the boundary token V - 1).  `verify` (optional dict: draft_probs,
    draft_tokens, temperature, bonus, vseed, vstep, n_accepted, next_token and
    pinned h_n_accepted / h_next_token) adds the speculative verify over the
    head's logits (logits_out required) to the captured step.  Every tensor
    passed must outlive the graph; the object keeps references to them.
    """

    def __init__(self, cache: KVCache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new,
                 attn_out, attn_ws, scale, W, ids, head_ws, h_inputs, d_inputs, h_ids,
                 h_boundary_count=None, causal=False, mode=TTS_ARGMAX, temperature=0.0, seed=None,
                 step=None, eos_allowed=None, best=None, logits_out=None, err=None, rope_base=0.0, verify=None):
        desc = _graph_desc(cache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new, attn_out,
                           attn_ws, scale, W, ids, head_ws, h_inputs, d_inputs, h_ids, h_boundary_count, causal,
                           mode, temperature, seed, step, eos_allowed, best, logits_out, err, rope_base, verify)
        self._verify = verify
        handle = ctypes.c_void_p()
        check("tts_step_graph_create", lib().tts_step_graph_create(ctypes.byref(desc), ctypes.byref(handle)))
        self._handle = handle
        self._keep = (cache, block_table, ctx_before, ctx_lens, q, k_new, v_new, attn_out, attn_ws, W, ids,
                      head_ws, h_inputs, d_inputs, h_ids, h_boundary_count, seed, step, eos_allowed, best,
                      logits_out, err)

    def launch(self, stream=None) -> None:
        if self._handle is None:
            raise ValueError("graph destroyed")
        check("tts_step_graph_launch", lib().tts_step_graph_launch(self._handle, _stream(stream)))

    def run(self, stream=None) -> None:
        """tts_step_graph_run: launch and return once the ids are in host memory."""
        if self._handle is None:
            raise ValueError("graph destroyed")
        check("tts_step_graph_run", lib().tts_step_graph_run(self._handle, _stream(stream)))

    def close(self) -> None:
        if getattr(self, "_handle", None) is not None:
            lib().tts_step_graph_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepGraphSet:
    """tts_step_graph_set_*: the step captured for several batch sizes.

    Takes StepGraph's arguments for the largest size (every per-stream tensor
    holding that many streams) plus `sizes` (increasing, the last the largest)
    and the packed input regions: `regions` is a list of (byte offset, bytes
    per stream) in h_inputs / d_inputs.  launch(n) runs the graph of the
    smallest size >= n and returns that size."""

    def __init__(self, cache: KVCache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new,
                 attn_out, attn_ws, scale, W, ids, head_ws, h_inputs, d_inputs, h_ids, sizes, regions,
                 h_boundary_count=None, causal=False, mode=TTS_ARGMAX, temperature=0.0, seed=None,
                 step=None, eos_allowed=None, best=None, logits_out=None, err=None, rope_base=0.0):
        desc = _graph_desc(cache, block_table, ctx_before, ctx_lens, max_ctx_len, q, k_new, v_new, attn_out,
                           attn_ws, scale, W, ids, head_ws, h_inputs, d_inputs, h_ids, h_boundary_count, causal,
                           mode, temperature, seed, step, eos_allowed, best, logits_out, err, rope_base)
        sz = (ctypes.c_int32 * len(sizes))(*[int(x) for x in sizes])
        off = (ctypes.c_size_t * len(regions))(*[int(o) for o, _ in regions])
        rb = (ctypes.c_size_t * len(regions))(*[int(b) for _, b in regions])
        handle = ctypes.c_void_p()
        check("tts_step_graph_set_create",
              lib().tts_step_graph_set_create(ctypes.byref(desc), sz, len(sizes), off, rb, len(regions),
                                              ctypes.byref(handle)))
        self._handle = handle
        self.sizes = [int(x) for x in sizes]
        self._keep = (cache, block_table, ctx_before, ctx_lens, q, k_new, v_new, attn_out, attn_ws, W, ids,
                      head_ws, h_inputs, d_inputs, h_ids, h_boundary_count, seed, step, eos_allowed, best,
                      logits_out, err)

    def launch(self, n_streams: int, stream=None) -> int:
        if self._handle is None:
            raise ValueError("graph set destroyed")
        chosen = ctypes.c_int32(0)
        check("tts_step_graph_set_launch",
              lib().tts_step_graph_set_launch(self._handle, int(n_streams), ctypes.byref(chosen), _stream(stream)))
        return chosen.value

    def run(self, n_streams: int, stream=None) -> int:
        """tts_step_graph_set_run: launch and return once the ids are in host
        memory; returns the size whose graph ran."""
        if self._handle is None:
            raise ValueError("graph set destroyed")
        chosen = ctypes.c_int32(0)
        check("tts_step_graph_set_run",
              lib().tts_step_graph_set_run(self._handle, int(n_streams), ctypes.byref(chosen), _stream(stream)))
        return chosen.value

    def close(self) -> None:
        if getattr(self, "_handle", None) is not None:
            lib().tts_step_graph_set_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class CodePredictor:
    """tts_code_predictor_*: the code predictor's frame loop on caller tensors.

    x0 [R][H], Wqkv [(Hq + 2 Hkv) * 128][H], W [n_steps][V][H], E
    [n_steps][V][H] (bf16, device); tokens int32 [n_steps][R] is written by
    each run.  The workspace is allocated here.  With graph=True the loop is
    captured once and run() launches the graph; multi_kernel=True runs one
    kernel per stage instead of the persistent kernel."""

    def __init__(self, x0, Wqkv, W, E, num_q_heads, num_kv_heads, tokens, mode=TTS_ARGMAX, temperature=0.0,
                 seed=None, step=None, err=None, graph=False, multi_kernel=False):
        R, H = x0.shape
        n_steps, V, HW = W.shape
        D = H // num_q_heads
        for t, n in ((x0, "x0"), (Wqkv, "Wqkv"), (W, "W"), (E, "E")):
            if t.dtype != torch.bfloat16:
                raise ValueError(f"{n} must be bfloat16")
        if HW != H or tuple(E.shape) != (n_steps, V, H) or Wqkv.shape[1] != H:
            raise ValueError("W and E must be [n_steps][V][H], Wqkv [F][H]")
        nbytes = lib().tts_code_predictor_workspace_size(R, H, num_q_heads, num_kv_heads, D, V, n_steps)
        if nbytes == 0:
            raise ValueError("unsupported code predictor shape")
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=x0.device)
        self.desc = _lib.CodePredictorDesc(
            R, H, num_q_heads, num_kv_heads, D, V, n_steps, int(mode), float(temperature), _dev(x0, "x0"),
            _dev(Wqkv, "Wqkv"), _dev(W, "W"), _dev(E, "E"), _keys(seed, "seed", R), _keys(step, "step", R),
            _dev(tokens, "tokens", torch.int32, (n_steps, R)), _dev(self.ws, "ws"), nbytes,
            None if err is None else _dev(err, "err", torch.int32), 1 if multi_kernel else 0)
        self._keep = (x0, Wqkv, W, E, tokens, seed, step, err)
        self._graph = None
        if graph:
            handle = ctypes.c_void_p()
            check("tts_code_predictor_graph_create",
                  lib().tts_code_predictor_graph_create(ctypes.byref(self.desc), ctypes.byref(handle)))
            self._graph = handle

    def run(self, stream=None) -> None:
        if self._graph is not None:
            check("tts_code_predictor_graph_launch", lib().tts_code_predictor_graph_launch(self._graph, _stream(stream)))
        else:
            check("tts_code_predictor_run", lib().tts_code_predictor_run(ctypes.byref(self.desc), _stream(stream)))

    def close(self) -> None:
        if getattr(self, "_graph", None) is not None:
            lib().tts_code_predictor_graph_destroy(self._graph)
            self._graph = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tts_status_string(code: int) -> str:
    return _lib.status_string(code)


def tts_version() -> int:
    return int(lib().tts_version())


def tts_set_launch_flags(flags: int) -> int:
    """Launch options of this thread's later single-kernel calls
    (_lib.LAUNCH_PROGRAMMATIC: programmatic dependents of the previous kernel
    in the stream).  Returns the previous flags."""
    return int(lib().tts_set_launch_flags(int(flags)))


def tts_test_set_stall(what: int, wait_limit_cycles: int = 2_000_000_000) -> None:
    """Test support: make a bounded on-device wait of the next kernels this
    thread launches run out (_lib.TEST_STALL_*), with the given wait limit."""
    check("tts_test_set_stall", lib().tts_test_set_stall(int(what), int(wait_limit_cycles)))


def tts_test_gumbel_noise(bits, out, stream=None) -> None:
    """Test support: the library's Gumbel noise of the 32-bit Philox words
    `bits` (int32 / uint32 view, device) into `out` (float32, same length)."""
    n = bits.numel()
    if out.numel() != n:
        raise ValueError("bits and out must have the same length")
    check("tts_test_gumbel_noise", lib().tts_test_gumbel_noise(_dev(bits, "bits", torch.int32), _dev(out, "out", torch.float32),
                                                               n, _stream(stream)))
