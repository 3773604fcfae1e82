"""Builds libttsdecode.so (the C-ABI library) in-tree for sm_103a.

    python -m decode_step_gb300.build [--force]

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library with the CUDA runtime linked statically, so the library loads
on a machine without a GPU (only its compute entry points need one).
"""
from __future__ import annotations

import argparse
import os
import platform
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["kv_append.cu", "decode_attn.cu", "head_select.cu", "spec_verify.cu", "tts_host.cpp",
           "tts_step.cpp", "tts_graph.cu", "code_predictor.cu"]


def lib_path() -> Path:
    return BUILD / f"libttsdecode_{platform.machine()}.so"


def nvcc() -> str:
    cand = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda")) / "bin" / "nvcc"
    return str(cand) if cand.exists() else "nvcc"


def _deps() -> list[Path]:
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + \
        list(INCLUDE.glob("*.h"))


def _compile(src: Path, obj: Path, verbose_ptxas: bool) -> None:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", str(INCLUDE), "-I", str(CSRC), "-c", str(src), "-o", str(obj)]
    if verbose_ptxas and src.suffix == ".cu":
        cmd += ["-Xptxas", "-v"]
    subprocess.run(cmd, check=True)


def build(force: bool = False, verbose_ptxas: bool = False) -> Path:
    out = lib_path()
    if not force and out.exists():
        newest = max(p.stat().st_mtime for p in _deps())
        if out.stat().st_mtime >= newest:
            return out
    objdir = BUILD / f"obj_{platform.machine()}"
    objdir.mkdir(parents=True, exist_ok=True)
    objs = [objdir / (Path(s).stem + ".o") for s in SOURCES]
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(lambda so: _compile(CSRC / so[0], so[1], verbose_ptxas),
                    zip(SOURCES, objs)))
    tmp = out.with_suffix(f".tmp{os.getpid()}.so")
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs),
                    "-cudart", "static", "-lpthread", "-ldl", "-lrt"], check=True)
    os.replace(tmp, out)
    return out


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true", help="print registers / spills per kernel")
    args = ap.parse_args()
    print(build(force=args.force, verbose_ptxas=args.ptxas_v))


if __name__ == "__main__":
    main()
