"""GB300 (sm_103a) batched decode step for streaming codec-LM text-to-speech.

C ABI: include/tts_decode.h (libttsdecode, built by `python -m
decode_step_gb300.build`).  `binding` mirrors the C functions for torch
tensors; `step.DecodeStep` chains append, attention and head for a batch.
"""
from ._lib import LibraryMissing, TTSError, declared_symbols, lib  # noqa: F401
