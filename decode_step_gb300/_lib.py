"""ctypes declarations of the C ABI in include/tts_decode.h.

Loads the in-tree libttsdecode built by `python -m decode_step_gb300.build`.
There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

from . import build as _build

TTS_OK = 0
TTS_F32, TTS_BF16, TTS_FP8_E4M3 = 0, 1, 2
TTS_ARGMAX, TTS_GUMBEL = 0, 1
TTS_VERIFY_BONUS = 1
ERRBIT_BLOCK_ID, ERRBIT_CTX_LEN, ERRBIT_TOKEN, ERRBIT_TIMEOUT = 1, 2, 4, 8
LAUNCH_PROGRAMMATIC = 1
TEST_STALL_NONE, TEST_STALL_ATTN_RING, TEST_STALL_PREDICTOR_GRID = 0, 1, 2

HEADER = Path(__file__).resolve().parents[1] / "include" / "tts_decode.h"

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_f32 = ctypes.c_float


class KVCacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", _i32), ("block_size", _i32), ("num_kv_heads", _i32),
                ("head_dim", _i32), ("dtype", _i32), ("k_pool", _vp), ("v_pool", _vp)]


class StepGraphDesc(ctypes.Structure):
    """tts_step_graph_desc."""
    _fields_ = [("cache", ctypes.POINTER(KVCacheDesc)), ("d_block_table", _vp), ("max_blocks_per_seq", _i32),
                ("d_ctx_before", _vp), ("d_ctx_lens", _vp), ("max_ctx_len", _i32), ("B", _i32), ("q_len", _i32),
                ("num_q_heads", _i32), ("scale", _f32), ("causal", _i32), ("rope_base", _f32), ("d_q", _vp), ("d_k_new", _vp),
                ("d_v_new", _vp), ("d_attn_out", _vp), ("d_attn_ws", _vp), ("attn_ws_bytes", _sz), ("d_W", _vp),
                ("V", _i32), ("mode", _i32), ("temperature", _f32), ("d_seed", _vp), ("d_step", _vp),
                ("d_eos_allowed", _vp), ("d_ids", _vp), ("d_best", _vp), ("d_logits_out", _vp),
                ("d_head_ws", _vp), ("head_ws_bytes", _sz), ("d_err", _vp), ("h_inputs", _vp), ("d_inputs", _vp),
                ("input_bytes", _sz), ("h_ids", _vp), ("h_boundary_count", _vp),
                ("d_draft_probs", _vp), ("d_draft_tokens", _vp), ("verify_temperature", _f32),
                ("verify_flags", _i32), ("d_vseed", _vp), ("d_vstep", _vp), ("d_n_accepted", _vp),
                ("d_next_token", _vp), ("h_n_accepted", _vp), ("h_next_token", _vp)]


class CodePredictorDesc(ctypes.Structure):
    """tts_code_predictor_desc."""
    _fields_ = [("R", _i32), ("H", _i32), ("num_q_heads", _i32), ("num_kv_heads", _i32), ("head_dim", _i32),
                ("V", _i32), ("n_steps", _i32), ("mode", _i32), ("temperature", _f32), ("d_x0", _vp),
                ("d_Wqkv", _vp), ("d_W", _vp), ("d_E", _vp), ("d_seed", _vp), ("d_step", _vp), ("d_tokens", _vp),
                ("d_ws", _vp), ("ws_bytes", _sz), ("d_err", _vp), ("flags", _i32)]


_SIGNATURES = {
    "tts_block_pool_create": (ctypes.c_int, [_i32, ctypes.POINTER(_vp)]),
    "tts_block_pool_alloc": (ctypes.c_int, [_vp, _i32, _vp]),
    "tts_block_pool_free": (ctypes.c_int, [_vp, _vp, _i32]),
    "tts_block_pool_num_free": (_i32, [_vp]),
    "tts_block_pool_destroy": (None, [_vp]),
    "tts_kv_append": (ctypes.c_int, [ctypes.POINTER(KVCacheDesc), _vp, _i32, _vp, _i32, _i32,
                                     _vp, _vp, _vp, _vp]),
    "tts_kv_append_rope": (ctypes.c_int, [ctypes.POINTER(KVCacheDesc), _vp, _i32, _vp, _i32, _i32, _i32,
                                          _f32, _vp, _vp, _vp, _vp, _vp]),
    "tts_decode_attn_workspace_size": (_sz, [_i32] * 6),
    "tts_decode_attn": (ctypes.c_int, [ctypes.POINTER(KVCacheDesc), _vp, _i32, _vp, _i32, _i32,
                                       _i32, _i32, _f32, _i32, _vp, _vp, _vp, _sz, _vp, _vp]),
    "tts_decode_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(KVCacheDesc), _vp, _i32, _vp, _i32,
                                               _i32, _i32, _i32, _f32, _i32, _vp, _vp, _vp, _vp]),
    "tts_head_workspace_size": (_sz, [_i32, _i32]),
    "tts_codebook_head_select": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32,
                                                _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tts_audio_head_select": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _i32,
                                             _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tts_spec_verify": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _f32, _vp, _vp, _i32,
                                       _vp, _vp, _vp, _vp]),
    "tts_decode_step": (ctypes.c_int, [ctypes.POINTER(KVCacheDesc), _vp, _i32, _vp, _vp, _i32, _i32,
                                       _i32, _i32, _f32, _i32, _f32, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                       _i32, _i32, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                       _vp, _vp]),
    "tts_step_graph_create": (ctypes.c_int, [ctypes.POINTER(StepGraphDesc), ctypes.POINTER(_vp)]),
    "tts_step_graph_launch": (ctypes.c_int, [_vp, _vp]),
    "tts_step_graph_run": (ctypes.c_int, [_vp, _vp]),
    "tts_step_graph_destroy": (None, [_vp]),
    "tts_step_graph_set_create": (ctypes.c_int, [ctypes.POINTER(StepGraphDesc), _vp, _i32, _vp, _vp, _i32,
                                                 ctypes.POINTER(_vp)]),
    "tts_step_graph_set_launch": (ctypes.c_int, [_vp, _i32, _vp, _vp]),
    "tts_step_graph_set_run": (ctypes.c_int, [_vp, _i32, _vp, _vp]),
    "tts_step_graph_set_destroy": (None, [_vp]),
    "tts_code_predictor_workspace_size": (_sz, [_i32] * 7),
    "tts_code_predictor_run": (ctypes.c_int, [ctypes.POINTER(CodePredictorDesc), _vp]),
    "tts_code_predictor_graph_create": (ctypes.c_int, [ctypes.POINTER(CodePredictorDesc), ctypes.POINTER(_vp)]),
    "tts_code_predictor_graph_launch": (ctypes.c_int, [_vp, _vp]),
    "tts_code_predictor_graph_destroy": (None, [_vp]),
    "tts_set_launch_flags": (_i32, [_i32]),
    "tts_test_set_stall": (ctypes.c_int, [_i32, ctypes.c_int64]),
    "tts_test_gumbel_noise": (ctypes.c_int, [_vp, _vp, _i32, _vp]),
    "tts_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tts_version": (ctypes.c_int, []),
}

_LIB = None


class LibraryMissing(RuntimeError):
    pass


def declared_symbols() -> list[str]:
    """Function names declared in include/tts_decode.h."""
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tts_[a-z0-9_]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """The loaded library (raises LibraryMissing if it was not built)."""
    global _LIB
    if _LIB is None:
        path = _build.lib_path()
        if not path.exists():
            raise LibraryMissing(f"{path} not built: run `python -m decode_step_gb300.build`")
        L = ctypes.CDLL(str(path))
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def status_string(code: int) -> str:
    return lib().tts_status_string(code).decode()


class TTSError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != TTS_OK:
        raise TTSError(fn, code)
