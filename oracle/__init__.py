"""CPU oracle for the batched codec-LM decode step.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's CPU
baseline call it; the product path never does.  It shares no code with the
CUDA library: the arithmetic lives in `tts_oracle.c` (plain C loops, sums in
double), and this module only compiles it with gcc and marshals numpy arrays.

Every function below follows the page passage cited in `tts_oracle.c`.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "tts_oracle.c"
BUILD_DIR = HERE / "_build"

_u8p = ctypes.POINTER(ctypes.c_uint8)
_vp = ctypes.c_void_p


def lib_path() -> Path:
    return BUILD_DIR / f"libtts_oracle_{platform.machine()}.so"


def build(src: Path | str = SRC, out: Path | str | None = None, force: bool = False) -> Path:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    out = Path(out) if out is not None else lib_path()
    src = Path(src)
    if not force and out.exists() and out.stat().st_mtime >= src.stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".tmp{os.getpid()}.so")
    cmd = ["gcc", "-std=gnu11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", str(tmp), str(src), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_vp)


class Oracle:
    """numpy front-end of one compiled oracle library."""

    def __init__(self, path: Path | str | None = None):
        path = Path(path) if path is not None else build()
        self.path = path
        L = ctypes.CDLL(str(path))
        L.orc_philox4x64_10.argtypes = [_vp, _vp, _vp]
        L.orc_philox4x64_10.restype = None
        L.orc_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                  ctypes.c_uint32, ctypes.c_uint32]
        L.orc_uniform.restype = ctypes.c_float
        L.orc_gumbel.argtypes = L.orc_uniform.argtypes
        L.orc_gumbel.restype = ctypes.c_float
        L.orc_kv_append.argtypes = [ctypes.c_int] * 4 + [_vp, _vp, _vp, ctypes.c_int, _vp,
                                                         ctypes.c_int, ctypes.c_int, _vp, _vp]
        L.orc_kv_append.restype = ctypes.c_int
        L.orc_decode_attn.argtypes = ([ctypes.c_int] * 4 + [_vp, _vp, _vp, ctypes.c_int, _vp]
                                      + [ctypes.c_int] * 3 + [ctypes.c_double, ctypes.c_int,
                                                              _vp, _vp])
        L.orc_decode_attn.restype = ctypes.c_int
        L.orc_head_select.argtypes = ([_vp, _vp] + [ctypes.c_int] * 5 + [ctypes.c_float]
                                      + [_vp] * 7)
        L.orc_head_select.restype = ctypes.c_int
        L.orc_spec_verify.argtypes = ([_vp, _vp, _vp] + [ctypes.c_int] * 3 + [ctypes.c_float]
                                      + [_vp, _vp, ctypes.c_int] + [_vp] * 4)
        L.orc_spec_verify.restype = ctypes.c_int
        L.orc_e4m3_encode_n.argtypes = [_vp, ctypes.c_size_t, _vp]
        L.orc_e4m3_encode_n.restype = None
        L.orc_e4m3_decode_n.argtypes = [_vp, ctypes.c_size_t, _vp]
        L.orc_e4m3_decode_n.restype = None
        L.orc_kv_append_fp8.argtypes = ([ctypes.c_int] * 3 + [_vp, _vp, ctypes.c_int, _vp]
                                        + [ctypes.c_int] * 2 + [_vp, _vp, ctypes.c_int])
        L.orc_rope_rows.argtypes = [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, ctypes.c_double, _vp]
        L.orc_rope_rows.restype = None
        L.orc_kv_append_fp8.restype = ctypes.c_int
        L.orc_decode_attn_fp8.argtypes = ([ctypes.c_int] * 3 + [_vp, _vp, ctypes.c_int, _vp]
                                          + [ctypes.c_int] * 3 + [ctypes.c_double, ctypes.c_int, _vp, _vp])
        L.orc_decode_attn_fp8.restype = ctypes.c_int
        L.orc_mish.argtypes = [ctypes.c_double]
        L.orc_mish.restype = ctypes.c_double
        L.orc_bf16_round.argtypes = [ctypes.c_double]
        L.orc_bf16_round.restype = ctypes.c_uint16
        L.orc_audio_expand.argtypes = [_vp, _vp, _vp] + [ctypes.c_int] * 3 + [_vp, _vp]
        L.orc_audio_expand.restype = ctypes.c_int
        L.orc_head_select_masked.argtypes = ([_vp, _vp, ctypes.c_int, _vp] + [ctypes.c_int] * 4
                                             + [ctypes.c_float, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp])
        L.orc_head_select_masked.restype = ctypes.c_int
        L.orc_code_predictor.argtypes = [ctypes.c_int] * 7 + [_vp] * 4 + [ctypes.c_int, ctypes.c_float] + [_vp] * 6
        L.orc_code_predictor.restype = ctypes.c_int
        self.lib = L

    # ------------------------------------------------------------- random
    def philox(self, ctr, key) -> np.ndarray:
        c = np.ascontiguousarray(ctr, dtype=np.uint64)
        k = np.ascontiguousarray(key, dtype=np.uint64)
        out = np.zeros(4, dtype=np.uint64)
        self.lib.orc_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
        return out

    def uniform(self, seed, step, tag, pos, idx) -> float:
        return float(self.lib.orc_uniform(int(seed), int(step), int(tag), int(pos), int(idx)))

    def gumbel(self, seed, step, tag, pos, idx) -> float:
        return float(self.lib.orc_gumbel(int(seed), int(step), int(tag), int(pos), int(idx)))

    # ------------------------------------------------------------- append
    def kv_append(self, k_pool, v_pool, block_table, ctx_before, k_new, v_new, inplace=False):
        """Writes k_new/v_new [B][q_len][Hkv][D] into the pools (into copies unless
        `inplace`, which needs C-contiguous arrays); returns them."""
        if not inplace:
            k_pool = np.array(k_pool, copy=True, order="C")
            v_pool = np.array(v_pool, copy=True, order="C")
        assert k_pool.flags["C_CONTIGUOUS"] and v_pool.flags["C_CONTIGUOUS"]
        num_blocks, Hkv, blk, D = k_pool.shape
        B, q_len = k_new.shape[:2]
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        cb = np.ascontiguousarray(ctx_before, dtype=np.int32)
        rc = self.lib.orc_kv_append(num_blocks, Hkv, D, k_pool.itemsize, _ptr(k_pool), _ptr(v_pool),
                                    _ptr(table), table.shape[1], _ptr(cb), B, q_len,
                                    _ptr(np.ascontiguousarray(k_new)),
                                    _ptr(np.ascontiguousarray(v_new)))
        if rc != 0:
            raise ValueError("oracle kv_append: slot outside the block table or pool")
        return k_pool, v_pool

    # ---------------------------------------------------------- attention
    def decode_attn(self, k_pool, v_pool, block_table, ctx_lens, q, scale, causal=False):
        """out[B][q_len][Hq][D] float64.  Pools are fp32 or bf16 bit patterns (uint16)."""
        is_bf16 = int(k_pool.dtype == np.uint16)
        num_blocks, Hkv, blk, D = k_pool.shape
        B, q_len, Hq, Dq = q.shape
        assert Dq == D and blk == 16 and Hq % Hkv == 0
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        L = np.ascontiguousarray(ctx_lens, dtype=np.int32)
        out = np.zeros((B, q_len, Hq, D), dtype=np.float64)
        rc = self.lib.orc_decode_attn(num_blocks, Hkv, D, is_bf16,
                                      _ptr(np.ascontiguousarray(k_pool)),
                                      _ptr(np.ascontiguousarray(v_pool)),
                                      _ptr(table), table.shape[1], _ptr(L), B, q_len, Hq,
                                      float(scale), int(bool(causal)),
                                      _ptr(np.ascontiguousarray(q)), _ptr(out))
        if rc != 0:
            raise ValueError("oracle decode_attn: invalid block id or context length")
        return out

    # ---------------------------------------------------------- FP8 cache
    def e4m3_encode(self, x) -> np.ndarray:
        """E4M3 codes (uint8) of float32 values: nearest, ties to even, +-448 saturation."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.zeros(x.shape, dtype=np.uint8)
        self.lib.orc_e4m3_encode_n(_ptr(x), x.size, _ptr(out))
        return out

    def e4m3_decode(self, c) -> np.ndarray:
        c = np.ascontiguousarray(c, dtype=np.uint8)
        out = np.zeros(c.shape, dtype=np.float32)
        self.lib.orc_e4m3_decode_n(_ptr(c), c.size, _ptr(out))
        return out

    def rope(self, x, pos, base=10000.0) -> np.ndarray:
        """Rotary embedding of rows x [..., D] (bf16 bits or float32) at positions
        pos (broadcast over x's leading dims); float32 result."""
        is_bf16 = int(x.dtype == np.uint16)
        xx = np.ascontiguousarray(x, dtype=np.uint16 if is_bf16 else np.float32)
        D = xx.shape[-1]
        rows = xx.size // D
        p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int32).reshape(
            np.asarray(pos).shape + (1,) * (xx.ndim - 1 - np.asarray(pos).ndim)), xx.shape[:-1])).reshape(rows)
        out = np.zeros(xx.shape, dtype=np.float32)
        self.lib.orc_rope_rows(_ptr(xx), is_bf16, rows, D, _ptr(np.ascontiguousarray(p, dtype=np.int32)),
                               float(base), _ptr(out))
        return out

    def kv_append_fp8(self, tiles, block_table, ctx_before, k_new, v_new):
        """FP8 append into a copy of the tile array (uint8 [num_blocks][Hkv][4224],
        the layout of orc_kv_append_fp8); k_new / v_new [B][q_len][Hkv][128] as
        bf16 bits (uint16) or float32.  Returns the new tiles."""
        t = np.array(tiles, dtype=np.uint8, copy=True, order="C")
        num_blocks, Hkv, nbytes = t.shape
        assert nbytes == 4224
        B, q_len, _, D = k_new.shape
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        cb = np.ascontiguousarray(ctx_before, dtype=np.int32)
        is_bf16 = int(k_new.dtype == np.uint16)
        assert v_new.dtype == k_new.dtype and k_new.dtype in (np.uint16, np.float32)
        rc = self.lib.orc_kv_append_fp8(num_blocks, Hkv, D, _ptr(t), _ptr(table), table.shape[1], _ptr(cb), B,
                                        q_len, _ptr(np.ascontiguousarray(k_new)), _ptr(np.ascontiguousarray(v_new)),
                                        is_bf16)
        if rc != 0:
            raise ValueError("oracle kv_append_fp8: slot outside the block table or pool")
        return t

    def decode_attn_fp8(self, tiles, block_table, ctx_lens, q, scale, causal=False):
        """out[B][q_len][Hq][128] float64 over an FP8 tile array; q bf16 bits."""
        num_blocks, Hkv, nbytes = tiles.shape
        B, q_len, Hq, D = q.shape
        assert nbytes == 4224 and D == 128 and Hq % Hkv == 0
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        L = np.ascontiguousarray(ctx_lens, dtype=np.int32)
        out = np.zeros((B, q_len, Hq, D), dtype=np.float64)
        rc = self.lib.orc_decode_attn_fp8(num_blocks, Hkv, D, _ptr(np.ascontiguousarray(tiles, dtype=np.uint8)),
                                          _ptr(table), table.shape[1], _ptr(L), B, q_len, Hq, float(scale),
                                          int(bool(causal)), _ptr(np.ascontiguousarray(q, dtype=np.uint16)),
                                          _ptr(out))
        if rc != 0:
            raise ValueError("oracle decode_attn_fp8: invalid block id or context length")
        return out

    # --------------------------------------------------------------- head
    def head_select(self, h, W, mode="argmax", T=0.0, seed=None, step=None,
                    eos_allowed=None, want_logits=False):
        """Returns dict(ids, best, second, logits?)."""
        is_bf16 = int(W.dtype == np.uint16)
        R, H = h.shape
        V, HW = W.shape
        assert HW == H and h.dtype == W.dtype
        m = {"argmax": 0, "gumbel": 1}[mode]
        if seed is None:
            seed = np.zeros(R, dtype=np.uint64)
        if step is None:
            step = np.zeros(R, dtype=np.uint64)
        seed = np.ascontiguousarray(seed, dtype=np.uint64)
        step = np.ascontiguousarray(step, dtype=np.uint64)
        eos = None if eos_allowed is None else np.ascontiguousarray(eos_allowed, dtype=np.uint8)
        ids = np.zeros(R, dtype=np.int32)
        best = np.zeros(R, dtype=np.float32)
        second = np.zeros(R, dtype=np.float32)
        logits = np.zeros((R, V), dtype=np.float32) if want_logits else None
        rc = self.lib.orc_head_select(_ptr(np.ascontiguousarray(h)), _ptr(np.ascontiguousarray(W)),
                                      is_bf16, R, H, V, m, float(T), _ptr(seed), _ptr(step),
                                      _ptr(eos), _ptr(ids), _ptr(best), _ptr(second), _ptr(logits))
        if rc != 0:
            raise ValueError("oracle head_select: bad arguments")
        out = dict(ids=ids, best=best, second=second)
        if want_logits:
            out["logits"] = logits
        return out

    # --------------------------------------------------------- audio head
    def mish(self, x) -> np.ndarray:
        """Mish of every element (float64)."""
        xs = np.asarray(x, dtype=np.float64)
        return np.vectorize(self.lib.orc_mish, otypes=[np.float64])(xs) if xs.size else xs.copy()

    def bf16_round(self, x) -> np.ndarray:
        """Nearest bfloat16 (ties to even) of float64 values, as uint16 bits."""
        xs = np.asarray(x, dtype=np.float64)
        return np.vectorize(self.lib.orc_bf16_round, otypes=[np.uint16])(xs) if xs.size else xs.astype(np.uint16)

    def audio_expand(self, h, W1, b1=None):
        """First audio-head layer: (z as bf16 bits [R][F], Mish values before rounding [R][F])."""
        R, H = h.shape
        F, HW = W1.shape
        assert HW == H and h.dtype == np.uint16 and W1.dtype == np.uint16
        z = np.zeros((R, F), dtype=np.uint16)
        m = np.zeros((R, F), dtype=np.float64)
        b = None if b1 is None else np.ascontiguousarray(b1, dtype=np.float32)
        rc = self.lib.orc_audio_expand(_ptr(np.ascontiguousarray(h)), _ptr(np.ascontiguousarray(W1)), _ptr(b),
                                       R, H, F, _ptr(z), _ptr(m))
        if rc != 0:
            raise ValueError("oracle audio_expand: bad arguments")
        return z, m

    def head_select_masked(self, h, W, b=None, mode="argmax", T=0.0, seed=None, step=None, n_tail=0,
                           tail_allowed=None, want_logits=False):
        """Head selection with bias b [V] and the last n_tail ids masked per row
        by tail_allowed [R] (uint32 bits).  Returns dict(ids, best, second, logits?)."""
        is_bf16 = int(W.dtype == np.uint16)
        R, H = h.shape
        V, HW = W.shape
        assert HW == H and h.dtype == W.dtype
        m = {"argmax": 0, "gumbel": 1}[mode]
        seed = np.zeros(R, np.uint64) if seed is None else np.ascontiguousarray(seed, dtype=np.uint64)
        step = np.zeros(R, np.uint64) if step is None else np.ascontiguousarray(step, dtype=np.uint64)
        bb = None if b is None else np.ascontiguousarray(b, dtype=np.float32)
        ta = None if tail_allowed is None else np.ascontiguousarray(tail_allowed, dtype=np.uint32)
        ids = np.zeros(R, dtype=np.int32)
        best = np.zeros(R, dtype=np.float32)
        second = np.zeros(R, dtype=np.float32)
        logits = np.zeros((R, V), dtype=np.float32) if want_logits else None
        rc = self.lib.orc_head_select_masked(_ptr(np.ascontiguousarray(h)), _ptr(np.ascontiguousarray(W)), is_bf16,
                                             _ptr(bb), R, H, V, m, float(T), _ptr(seed), _ptr(step), int(n_tail),
                                             _ptr(ta), _ptr(ids), _ptr(best), _ptr(second), _ptr(logits))
        if rc != 0:
            raise ValueError("oracle head_select_masked: bad arguments")
        out = dict(ids=ids, best=best, second=second)
        if want_logits:
            out["logits"] = logits
        return out

    def audio_head(self, h, W1, b1, W2, b2, mode="argmax", T=0.0, seed=None, step=None, n_tail=0,
                   tail_allowed=None, want_logits=False):
        """The two-layer audio head: z = bf16(Mish(h W1^T + b1)), then the masked
        selection over z W2^T + b2.  Returns the selection dict plus z."""
        z, _ = self.audio_expand(h, W1, b1)
        out = self.head_select_masked(z, W2, b2, mode, T, seed, step, n_tail, tail_allowed, want_logits)
        out["z"] = z
        return out

    # ----------------------------------------------------- code predictor
    def code_predictor(self, x0, Wqkv, W, E, Hq, Hkv, mode="argmax", T=0.0, seed=None, step=None,
                       want_trace=False):
        """The code predictor's frame loop.  x0 [R][H], Wqkv [(Hq+2Hkv)D][H],
        W [n_steps][V][Hq D], E [n_steps][V][H], all bf16 bits.  Returns
        dict(tokens, best, second) [n_steps][R] and, with want_trace, trace
        [n_steps][R][(Hq+2Hkv)D + Hq D] (bf16 values of q, k, v, o)."""
        R, H = x0.shape
        F = Wqkv.shape[0]
        n_steps, V, HO = W.shape
        D = HO // Hq
        assert F == (Hq + 2 * Hkv) * D and E.shape == (n_steps, V, H) and Wqkv.shape[1] == H
        m = {"argmax": 0, "gumbel": 1}[mode]
        seed = np.zeros(R, np.uint64) if seed is None else np.ascontiguousarray(seed, dtype=np.uint64)
        step = np.zeros(R, np.uint64) if step is None else np.ascontiguousarray(step, dtype=np.uint64)
        tokens = np.zeros((n_steps, R), np.int32)
        best = np.zeros((n_steps, R), np.float32)
        second = np.zeros((n_steps, R), np.float32)
        trace = np.zeros((n_steps, R, F + HO), np.float64) if want_trace else None
        rc = self.lib.orc_code_predictor(R, H, Hq, Hkv, D, V, n_steps, _ptr(np.ascontiguousarray(x0)),
                                         _ptr(np.ascontiguousarray(Wqkv)), _ptr(np.ascontiguousarray(W)),
                                         _ptr(np.ascontiguousarray(E)), m, float(T), _ptr(seed), _ptr(step),
                                         _ptr(tokens), _ptr(best), _ptr(second), _ptr(trace))
        if rc != 0:
            raise ValueError("oracle code_predictor: bad arguments")
        out = dict(tokens=tokens, best=best, second=second)
        if want_trace:
            out["trace"] = trace
        return out

    # ------------------------------------------------------------- verify
    def spec_verify(self, target_logits, draft_probs, draft_tokens, T, seed, step, bonus=False):
        """Returns dict(n_accepted, next_token, gap_accept, gap_resid)."""
        tl = np.ascontiguousarray(target_logits, dtype=np.float32)
        dp = np.ascontiguousarray(draft_probs, dtype=np.float32)
        dt = np.ascontiguousarray(draft_tokens, dtype=np.int32)
        B, K1, V = tl.shape
        K = K1 - 1
        assert dp.shape == (B, K, V) and dt.shape == (B, K)
        seed = np.ascontiguousarray(seed, dtype=np.uint64)
        step = np.ascontiguousarray(step, dtype=np.uint64)
        n_acc = np.zeros(B, dtype=np.int32)
        nxt = np.zeros(B, dtype=np.int32)
        ga = np.zeros(B, dtype=np.float32)
        gr = np.zeros(B, dtype=np.float32)
        rc = self.lib.orc_spec_verify(_ptr(tl), _ptr(dp), _ptr(dt), B, K, V, float(T),
                                      _ptr(seed), _ptr(step), int(bool(bonus)),
                                      _ptr(n_acc), _ptr(nxt), _ptr(ga), _ptr(gr))
        if rc != 0:
            raise ValueError("oracle spec_verify: draft token outside the vocabulary")
        return dict(n_accepted=n_acc, next_token=nxt, gap_accept=ga, gap_resid=gr)


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    """The oracle built from `tts_oracle.c` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
