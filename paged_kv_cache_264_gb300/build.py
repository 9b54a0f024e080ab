"""Build ``libpagedkv.so`` from ``csrc/`` with nvcc for sm_103a (in-tree, under
``_build/<machine>/``).  Translation units compile in parallel; a unit is rebuilt only
when it or a header is newer than its object file."""

from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
ROOT = PKG.parent
INCLUDE = ROOT / "include"
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["pkv_api.cu", "pkv_cache.cu", "pkv_decode_bf16.cu", "pkv_decode_int8.cu",
           "pkv_decode_fp8.cu", "pkv_decode_mma.cu", "pkv_decode_mma_bf16.cu", "pkv_decode_mma_int8.cu",
           "pkv_decode_mma_fp8.cu", "pkv_decode_mma_quant_d64.cu", "pkv_static_scratch.cu", "pkv_selftest.cu", "pkv_blocks.cpp"]


def build_dir() -> Path:
    return PKG / "_build" / platform.machine()


def library_path() -> Path:
    return build_dir() / "libpagedkv.so"


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _headers_mtime() -> float:
    hs = list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h"))
    return max((h.stat().st_mtime for h in hs), default=0.0)


def compile_flags(extra: list[str] | None = None) -> list[str]:
    return [
        *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
        "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}", f"-I{CSRC}",
        "--expt-relaxed-constexpr", *(extra or []),
    ]


def _compile(src: Path, obj: Path, extra: list[str] | None, verbose: bool) -> None:
    cmd = [nvcc(), *compile_flags(extra), "-c", str(src), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src.name}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> Path:
    out = library_path()
    bdir = build_dir()
    bdir.mkdir(parents=True, exist_ok=True)
    hdr = _headers_mtime()
    jobs = []
    objs = []
    for name in SOURCES:
        src = CSRC / name
        obj = bdir / (Path(name).stem + ".o")
        objs.append(obj)
        stale = force or not obj.exists() or obj.stat().st_mtime < max(src.stat().st_mtime, hdr)
        if stale:
            jobs.append((src, obj))
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(lambda j: _compile(j[0], j[1], extra, verbose), jobs))
    if jobs or not out.exists():
        tmp = out.with_suffix(f".{os.getpid()}.tmp")
        cmd = [nvcc(), *ARCH_FLAGS, "-shared", "-o", str(tmp), *map(str, objs), "-lcudart_static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    p = build(force="--force" in sys.argv, verbose=True)
    print(p)
