"""Build the C-ABI shared library libtgemm.so for sm_103a, in-tree.

Each .cu translation unit is compiled by nvcc in parallel into
``_build/*.o`` and linked into ``_build/libtgemm.so`` (static CUDA runtime,
only the ``tgemm_*`` symbols exported).  A unit is rebuilt when it, any
header or the flags changed.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libtgemm.so")

SOURCES = [
    "tgemm_api.cu",
    "tgemm_inst_f16.cu",
    "tgemm_inst_bf16.cu",
    "tgemm_inst_f32.cu",
    "tgemm_debug.cu",
    "tgemm_noalloc.cu",
]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                 "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtgemm.so")
    return cand


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh", ".inc"))]
    hs.append(os.path.join(INCLUDE, "tgemm.h"))
    return sorted(hs)


def _digest(src: str, extra_flags) -> str:
    h = hashlib.sha256()
    for path in [src] + _headers():
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(CFLAGS + list(extra_flags)).encode())
    return h.hexdigest()


def _compile(src_name: str, extra_flags, verbose: bool):
    src = os.path.join(CSRC, src_name)
    obj = os.path.join(OUT, src_name.replace(".cu", ".o"))
    stamp = obj + ".sha256"
    dig = _digest(src, extra_flags)
    if os.path.exists(obj) and os.path.exists(stamp) and open(stamp).read() == dig:
        return obj, False
    cmd = [_nvcc()] + CFLAGS + list(extra_flags) + ["-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src_name, " ".join(cmd), r.stderr))
    if verbose and r.stderr:
        print(r.stderr)
    os.replace(obj + ".tmp", obj)
    with open(stamp, "w") as f:
        f.write(dig)
    return obj, True


def build(verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libtgemm.so if anything changed; return its path."""
    os.makedirs(OUT, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra_flags, verbose), SOURCES))
    objs = [o for o, _ in results]
    relink = any(changed for _, changed in results) or not os.path.exists(LIB)
    if relink:
        tmp = LIB + ".tmp"
        cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-ldl", "-lpthread",
                                                                  "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv))
