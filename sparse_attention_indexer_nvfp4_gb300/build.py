"""Build libidx.so (the C-ABI library) in-tree for sm_103a with nvcc.

    python -m sparse_attention_indexer_nvfp4_gb300.build

Each .cu under csrc/ compiles to an object in _build/ (in parallel), then
nvcc links them into _lib/libidx.so with the CUDA runtime linked statically.
A one-line probe decides IDX_HAVE_QMUL4: whether this toolchain's ptxas
accepts mul.rn.satfinite.e4m3x4.e2m1x4.e4m3x4 (it needs a newer ptxas than
CUDA 13.0's); without it the exact fp32-then-round-once dequant is used.
"""

from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libidx.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def probe_qmul4() -> bool:
    src = (
        "#include <cstdint>\n__global__ void k(const uint32_t* s, const uint16_t* c, uint32_t* o) {\n"
        "  uint32_t r;\n  asm volatile(\"mul.rn.satfinite.e4m3x4.e2m1x4.e4m3x4 %0, %1, %2;\" : \"=r\"(r) : "
        "\"h\"(c[0]), \"r\"(s[0]));\n  o[0] = r;\n}\n"
    )
    with tempfile.TemporaryDirectory() as d:
        p = os.path.join(d, "q.cu")
        with open(p, "w") as f:
            f.write(src)
        r = subprocess.run([nvcc(), *ARCH, "-c", p, "-o", os.path.join(d, "q.o")], capture_output=True, text=True)
        return r.returncode == 0


def _flags(qmul4: bool) -> list[str]:
    return [
        *ARCH,
        "-O3",
        "-lineinfo",
        "-std=c++17",
        "-Xcompiler",
        "-fPIC",
        "-Xptxas",
        "-v" if os.environ.get("IDX_PTXAS_VERBOSE") else "-O3",
        f"-DIDX_HAVE_QMUL4={1 if qmul4 else 0}",
        "-I",
        INCLUDE,
        "-I",
        CSRC,
    ]


def _compile(src: str, obj: str, flags: list[str]) -> tuple[str, int, str]:
    r = subprocess.run([nvcc(), *flags, "-c", src, "-o", obj], capture_output=True, text=True)
    return src, r.returncode, r.stdout + r.stderr


def _stamp(flags: list[str]) -> str:
    h = hashlib.sha256(" ".join(flags).encode())
    for name in sorted(os.listdir(CSRC)) + ["idx.h"]:
        path = os.path.join(CSRC, name) if name != "idx.h" else os.path.join(INCLUDE, name)
        with open(path, "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link; returns the library path.  Skips work when nothing changed."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    qmul4 = probe_qmul4()
    flags = _flags(qmul4)
    stamp = _stamp(flags)
    stamp_file = os.path.join(BUILD, "libidx.stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return LIB
    sources = sorted(os.path.join(CSRC, n) for n in os.listdir(CSRC) if n.endswith(".cu"))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in sources]
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        results = list(ex.map(lambda so: _compile(so[0], so[1], flags), zip(sources, objs)))
    failed = [(s, out) for s, rc, out in results if rc != 0]
    for s, rc, out in results:
        if verbose and out.strip():
            print(f"--- {os.path.basename(s)}\n{out}")
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"{s}:\n{out}" for s, out in failed))
    tmp = LIB + ".tmp"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    if verbose:
        print(f"built {LIB} (QMUL4 {'on' if qmul4 else 'off'})")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
