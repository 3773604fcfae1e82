"""The C-ABI library on the host: it loads without a GPU, exports every
declared symbol, runs the block pool, and rejects bad arguments before
launching anything (CPU only; no compute call is made)."""
import ctypes

import pytest

import decode_step_gb300 as pkg
from decode_step_gb300 import _lib
from decode_step_gb300.build import build


@pytest.fixture(scope="module")
def L():
    build()
    return pkg.lib()


def test_exports_every_declared_symbol(L):
    names = pkg.declared_symbols()
    assert len(names) >= 13
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert L.tts_version() >= 100


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5):
        assert L.tts_status_string(code)
    assert L.tts_status_string(-99) == b"unknown status"


def test_block_pool_lifo_all_or_nothing(L):
    from decode_step_gb300.binding import BlockPool, TTSError
    p = BlockPool(8)
    a = p.alloc(3)
    assert a == [0, 1, 2] and p.num_free == 5
    with pytest.raises(TTSError) as e:
        p.alloc(6)
    assert e.value.code == -5 and p.num_free == 5     # exhausted, nothing taken
    p.free([1])
    assert p.alloc(1) == [1]                          # last freed, first reused
    with pytest.raises(TTSError):
        p.free([0, 0])                                # repeated id
    with pytest.raises(TTSError):
        p.free([2, 7])                                # 7 was never handed out
    with pytest.raises(TTSError):
        p.free([9])                                   # outside the pool
    assert p.num_free == 5                            # failed frees changed nothing
    p.free([0, 1, 2])
    assert p.num_free == 8
    assert sorted(p.alloc(8)) == list(range(8))
    p.close()


def test_block_pool_rejects_bad_create(L):
    h = ctypes.c_void_p()
    assert L.tts_block_pool_create(0, ctypes.byref(h)) == -1
    assert L.tts_block_pool_create(5, None) == -1
    assert L.tts_block_pool_num_free(None) == -1


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: every call below fails validation first


def _cache(num_blocks=8, hkv=8, d=128, dtype=1, block=16):
    return _lib.KVCacheDesc(num_blocks, block, hkv, d, dtype, FAKE, FAKE)


def test_workspace_queries(L):
    assert L.tts_decode_attn_workspace_size(64, 1, 16, 8, 128, 1500) > 0
    assert L.tts_decode_attn_workspace_size(64, 1, 15, 8, 128, 1500) == 0   # Hq % Hkv
    assert L.tts_decode_attn_workspace_size(64, 9, 16, 8, 128, 1500) == 0   # 18 query rows
    assert L.tts_head_workspace_size(0, 10) == 0
    assert L.tts_head_workspace_size(64, 4097) >= 64 * 8


def test_attention_argument_checks(L):
    c = _cache()
    args = lambda **k: dict(dict(cache=ctypes.byref(c), table=FAKE, maxb=94, ctx=FAKE, maxctx=1500,  # noqa: E731
                                  B=4, q_len=1, Hq=16, scale=0.08, causal=0, q=FAKE, out=FAKE,
                                  ws=FAKE, wsb=0, err=None, stream=None), **k)
    def call(**k):
        a = args(**k)
        return L.tts_decode_attn(a["cache"], a["table"], a["maxb"], a["ctx"], a["maxctx"], a["B"],
                                 a["q_len"], a["Hq"], a["scale"], a["causal"], a["q"], a["out"],
                                 a["ws"], a["wsb"], a["err"], a["stream"])
    assert call(q=None) == -1
    assert call(Hq=12) == -1                      # not a multiple of Hkv
    assert call(scale=-1.0) == -1
    assert call(q_len=9) == -2                    # 18 rows per KV head
    bad = _cache(d=96)
    assert call(cache=ctypes.byref(bad)) == -2
    bad = _cache(block=32)
    assert call(cache=ctypes.byref(bad)) == -2
    assert call(wsb=16) == -3                     # workspace too small
    assert call(B=0, wsb=0) == 0                  # nothing to do


def test_append_head_verify_argument_checks(L):
    c = _cache()
    assert L.tts_kv_append(ctypes.byref(c), FAKE, 4, None, 2, 1, FAKE, FAKE, None, None) == -1
    assert L.tts_kv_append(ctypes.byref(c), FAKE, 4, FAKE, 2, 0, FAKE, FAKE, None, None) == -1
    assert L.tts_kv_append(ctypes.byref(c), FAKE, 4, FAKE, 0, 1, FAKE, FAKE, None, None) == 0
    head = lambda **k: L.tts_codebook_head_select(  # noqa: E731
        k.get("h", FAKE), FAKE, k.get("dtype", 1), k.get("R", 4), k.get("H", 2048),
        k.get("V", 4097), k.get("mode", 0), k.get("T", 0.0), k.get("seed", None), None, None,
        FAKE, None, None, k.get("ws", FAKE), k.get("wsb", 0), None)
    assert head(h=None) == -1
    assert head(R=0) == -1
    assert head(mode=1) == -1                     # Gumbel needs seeds and T > 0
    assert head(dtype=5) == -2
    assert head() == -3                           # workspace too small
    assert head(H=100, wsb=1 << 20) == -2         # bf16 tensor-core path needs H % 64 == 0
    ver = lambda **k: L.tts_spec_verify(  # noqa: E731
        FAKE, FAKE, FAKE, 4, k.get("K", 4), 97, k.get("T", 0.7), FAKE, FAKE, k.get("flags", 0),
        FAKE, FAKE, None, None)
    assert ver(K=0) == -1 and ver(K=17) == -1 and ver(T=0.0) == -1 and ver(flags=2) == -1


def test_struct_layouts_match_header(tmp_path):
    """The ctypes mirrors of tts_kv_cache, tts_step_graph_desc and
    tts_code_predictor_desc have the C layout the header gives (compiled here
    against the header)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f for f, _ in _lib.StepGraphDesc._fields_]
    pfields = [f for f, _ in _lib.CodePredictorDesc._fields_]
    src = ["#include <stdio.h>", "#include <stddef.h>", '#include "tts_decode.h"', "int main(void) {",
           'printf("%zu %zu\\n", sizeof(tts_kv_cache), offsetof(tts_kv_cache, v_pool));',
           'printf("%zu\\n", sizeof(tts_step_graph_desc));']
    src += [f'printf("%zu\\n", offsetof(tts_step_graph_desc, {f}));' for f in fields]
    src += ['printf("%zu\\n", sizeof(tts_code_predictor_desc));']
    src += [f'printf("%zu\\n", offsetof(tts_code_predictor_desc, {f}));' for f in pfields]
    src += ["return 0; }"]
    (tmp_path / "lay.c").write_text("\n".join(src) + "\n")
    subprocess.run([cc, "-I", str(_lib.HEADER.parent), "-o", str(tmp_path / "lay"), str(tmp_path / "lay.c")],
                   check=True)
    out = subprocess.run([str(tmp_path / "lay")], capture_output=True, text=True, check=True).stdout.split()
    vals = [int(x) for x in out]
    K = _lib.KVCacheDesc
    assert vals[:2] == [ctypes.sizeof(K), K.v_pool.offset]
    assert vals[2] == ctypes.sizeof(_lib.StepGraphDesc)
    n = 3 + len(fields)
    assert vals[3:n] == [getattr(_lib.StepGraphDesc, f).offset for f in fields]
    P = _lib.CodePredictorDesc
    assert vals[n] == ctypes.sizeof(P)
    assert vals[n + 1:] == [getattr(P, f).offset for f in pfields]


def test_step_graph_rejects_bad_descriptors(L):
    handle = ctypes.c_void_p()
    assert L.tts_step_graph_create(None, ctypes.byref(handle)) == -1
    desc = _lib.StepGraphDesc()  # all null
    assert L.tts_step_graph_create(ctypes.byref(desc), ctypes.byref(handle)) == -1
    assert L.tts_step_graph_launch(None, None) == -1
    assert L.tts_step_graph_run(None, None) == -1
    chosen = ctypes.c_int32(-7)
    assert L.tts_step_graph_set_run(None, 4, ctypes.byref(chosen), None) == -1
    assert chosen.value == -7                         # nothing chosen for a missing set
    L.tts_step_graph_destroy(None)


def test_rope_append_and_noalloc_attention_argument_checks(L):
    c = _cache()
    rope = lambda **k: L.tts_kv_append_rope(  # noqa: E731
        ctypes.byref(k.get("cache", c)), FAKE, 4, FAKE, k.get("B", 2), 1, k.get("Hq", 16),
        k.get("base", 10000.0), k.get("q", FAKE), FAKE, FAKE, None, None)
    assert rope(base=0.0) == -1                       # the plain append is tts_kv_append
    assert rope(base=1.0) == -1 and rope(base=float("inf")) == -1
    assert rope(q=None) == -1
    assert rope(Hq=12) == -1                          # not a multiple of Hkv
    assert rope(cache=_cache(dtype=0, d=64)) == -2    # fp32 rows have no rotary build
    assert rope(cache=_cache(d=64)) == -2
    assert rope(B=0) == 0                             # nothing to do
    noalloc = lambda **k: L.tts_decode_attn_noalloc(  # noqa: E731
        k.get("cache", ctypes.byref(c)), FAKE, 94, FAKE, 1500, k.get("B", 4), 1, k.get("Hq", 16), 0.08, 0,
        k.get("q", FAKE), FAKE, None, None)
    assert noalloc(cache=None) == -1
    assert noalloc(Hq=12) == -1                       # rejected before the static scratch is looked up
    assert noalloc(B=0) == 0


def test_audio_head_argument_checks(L):
    def audio(**k):
        return L.tts_audio_head_select(
            k.get("h", FAKE), FAKE, None, FAKE, None, k.get("R", 4), 2048, k.get("F", 4096), 4097, 1, None,
            k.get("mode", 0), 0.0, None, None, k.get("z", FAKE), FAKE, None, None, FAKE, 0, None)
    assert audio(mode=5) == -1
    assert audio(F=100) == -2                         # the second layer reduces over F: F % 64 == 0
    assert audio(F=0) == -2
    assert audio(h=None) == -1
    assert audio(z=None) == -1                        # the first layer writes z
    assert audio(R=0) == -1 and audio(R=5000) == -1


def test_code_predictor_argument_checks(L):
    assert L.tts_code_predictor_workspace_size(64, 1024, 8, 4, 128, 2048, 15) > 0
    assert L.tts_code_predictor_workspace_size(0, 1024, 8, 4, 128, 2048, 15) == 0
    assert L.tts_code_predictor_workspace_size(64, 1024, 8, 4, 128, 2048, 0) == 0

    def desc(**k):
        f = dict(R=64, H=1024, num_q_heads=8, num_kv_heads=4, head_dim=128, V=2048, n_steps=15, mode=0,
                 temperature=0.0, d_x0=FAKE.value, d_Wqkv=FAKE.value, d_W=FAKE.value, d_E=FAKE.value,
                 d_seed=None, d_step=None, d_tokens=FAKE.value, d_ws=FAKE.value, ws_bytes=0, d_err=None, flags=0)
        f.update(k)
        return _lib.CodePredictorDesc(**f)
    run = lambda **k: L.tts_code_predictor_run(ctypes.byref(desc(**k)), None)  # noqa: E731
    assert L.tts_code_predictor_run(None, None) == -1
    assert run(d_x0=None) == -1
    assert run(R=0) == -1
    assert run(num_q_heads=6) == -1                   # not a multiple of the KV heads
    assert run(num_q_heads=12) == -2                  # heads x head_dim must equal H
    assert run() == -3                                # workspace too small
    handle = ctypes.c_void_p()
    assert L.tts_code_predictor_graph_create(ctypes.byref(desc(d_E=None)), ctypes.byref(handle)) == -1
    assert L.tts_code_predictor_graph_launch(None, None) == -1
    L.tts_code_predictor_graph_destroy(None)


def test_step_graph_set_rejects_bad_sizes(L):
    desc = _lib.StepGraphDesc()
    desc.B = 64
    desc.input_bytes = 64 * 1024
    handle = ctypes.c_void_p()
    i32 = lambda *v: (ctypes.c_int32 * len(v))(*v)    # noqa: E731
    sz = lambda *v: (ctypes.c_size_t * len(v))(*v)    # noqa: E731

    def create(sizes, offs=(0,), rows=(16,), d=desc):
        s = i32(*sizes) if sizes else None
        return L.tts_step_graph_set_create(ctypes.byref(d) if d is not None else None, s, len(sizes),
                                           sz(*offs), sz(*rows), len(offs), ctypes.byref(handle))
    assert create([1, 4, 64], d=None) == -1
    assert create([]) == -1                            # no size
    assert create(list(range(1, 18))) == -1            # more than TTS_GRAPH_SET_MAX sizes
    assert create([4, 4, 64]) == -1                    # not strictly increasing
    assert create([1, 4, 32]) == -1                    # the largest size must be B
    assert create([1, 4, 65]) == -1                    # beyond B
    assert create([1, 64], offs=(8,)) == -1            # a region not 16-byte aligned
    assert create([1, 64], rows=(6,)) == -1            # row bytes not a multiple of 4
    assert create([1, 64], rows=(2048,)) == -1         # B rows of 2 KB overrun 64 KB
    assert create([1, 64], offs=(64 * 1024,)) == -1    # starts past the buffers
    assert L.tts_step_graph_set_launch(None, 4, None, None) == -1
    L.tts_step_graph_set_destroy(None)


def test_launch_flags_and_stall_arguments():
    """The thread's launch flags round-trip; the test stall rejects unknown
    modes and wait limits outside [1e3, 4e9] (host-side checks, no GPU)."""
    from decode_step_gb300 import _lib
    lib = _lib.lib()
    prev = lib.tts_set_launch_flags(_lib.LAUNCH_PROGRAMMATIC)
    assert lib.tts_set_launch_flags(prev) == _lib.LAUNCH_PROGRAMMATIC
    assert lib.tts_set_launch_flags(0) == prev
    assert lib.tts_test_set_stall(3, 10_000) == -1
    assert lib.tts_test_set_stall(1, 10) == -1
    assert lib.tts_test_set_stall(1, 5_000_000_000) == -1
    assert lib.tts_test_set_stall(0, 2_000_000_000) == 0


def test_gumbel_noise_arguments():
    """The Gumbel-noise test entry point rejects a negative count and null
    pointers, and does nothing for n = 0 (host-side checks, no GPU)."""
    from decode_step_gb300 import _lib
    lib = _lib.lib()
    assert lib.tts_test_gumbel_noise(None, None, 4, None) == -1
    assert lib.tts_test_gumbel_noise(None, None, -1, None) == -1
    assert lib.tts_test_gumbel_noise(None, None, 0, None) == 0
