"""Build libmla.so in-tree with nvcc for sm_103a.

    python -m head_latent_attention_29_b300._build [--force]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
LIB_PATH = os.path.join(PKG_DIR, "libmla.so")
INCLUDE = os.path.join(os.path.dirname(PKG_DIR), "include")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-shared",
]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: cannot build libmla")


def _sources() -> list[str]:
    out = [os.path.join(INCLUDE, "mla.h")]
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            out.append(os.path.join(CSRC, name))
    return out


def source_hash() -> str:
    """sha256[:16] over the library's sources (header and csrc, names and bytes); the
    build compiles it into the library, which reports it through
    mla_build_source_hash(), so a library built from other sources is recognised
    whatever the files' times."""
    import hashlib
    h = hashlib.sha256()
    for path in _sources():
        h.update(os.path.relpath(path, os.path.dirname(PKG_DIR)).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def built_hash(path: str = LIB_PATH) -> str | None:
    """The source hash compiled into the library file at `path` (None if it has
    none).  Read from the file's bytes (the tagged string mla_build_source_hash
    returns), not by loading it: a process that loaded the old file would get that
    one back from the loader after a rebuild."""
    import re
    try:
        with open(path, "rb") as f:
            m = re.search(rb"MLA-SOURCE-HASH:([0-9a-f]{16}|unknown)", f.read())
    except OSError:
        return None
    return m.group(1).decode() if m else None


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    return built_hash() != source_hash()


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB_PATH
    tmp = LIB_PATH + ".tmp"
    cmd = [_nvcc(), *NVCC_FLAGS, f"-DMLA_SOURCE_HASH=\"{source_hash()}\"", os.path.join(CSRC, "libmla.cu"), "-o", tmp]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
