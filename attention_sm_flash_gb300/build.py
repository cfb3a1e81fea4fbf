"""Builds libattn.so in-tree from csrc/*.cu for sm_103a with nvcc (no cmake, no torch).

Each translation unit is compiled in parallel to an object under ``_build/``; the
objects are linked into ``_lib/libattn.so`` (cudart linked statically, so the library
needs only the CUDA driver at run time). Rebuilds only when a source, a header or the
flags changed.

    python -m attention_sm_flash_gb300.build [--force] [--verbose]
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stamp(extra_flags) -> str:
    h = hashlib.sha256()
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra_flags)).encode())
    files = _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h")) +
                                glob.glob(os.path.join(CSRC, "*.cuh")) +
                                glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in files:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def _code_text(src: bytes) -> bytes:
    """The code of a C/C++/CUDA source without its comments, with every run of whitespace
    made one space: what source_digest covers, so that editing a comment or the layout of
    a file leaves the digest (and the figures recorded under it) as they were. String and
    character literals are kept whole, comment markers inside them included."""
    out = bytearray()
    i, n = 0, len(src)
    while i < n:
        c = src[i]
        if c in b"\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == 0x5C else 1  # a backslash escapes the next byte
            out += src[i:j + 1]
            i = j + 1
        elif src.startswith(b"//", i):
            j = src.find(b"\n", i)
            i = n if j < 0 else j
            out += b" "
        elif src.startswith(b"/*", i):
            j = src.find(b"*/", i + 2)
            i = n if j < 0 else j + 2
            out += b" "
        else:
            out.append(c)
            i += 1
    return b" ".join(bytes(out).split())


def source_digest(kernel_files=None) -> str:
    """Hash of the code (comments and layout aside) of the CUDA sources and headers, by
    relative path (the same on any machine and checkout path): the key under which
    measured per-kernel figures, such as DRAM traffic, are recorded. ``kernel_files``:
    names of the .cu files that hold the measured kernels (with every header, the code
    they include); None = all sources."""
    h = hashlib.sha256()
    sources = _sources()
    if kernel_files is not None:
        sources = [f for f in sources if os.path.basename(f) in set(kernel_files)]
    files = sources + sorted(glob.glob(os.path.join(CSRC, "*.h")) +
                             glob.glob(os.path.join(CSRC, "*.cuh")) +
                             glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in sorted(files, key=lambda p: os.path.relpath(p, ROOT)):
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, "rb") as fh:
            h.update(_code_text(fh.read()))
    return h.hexdigest()[:16]


# the source file of each operation's kernels by element type, for per-kernel digests
OP_SOURCES = {
    ("attn_fwd", "bf16"): ["fwd_sm103.cu"],
    ("attn_fwd", "f32"): ["fwd_tf32x3.cu"],
    ("attn_fwd_paged", "bf16"): ["fwd_sm103.cu"],
    ("attn_fwd_splitkv", "bf16"): ["fwd_sm103.cu"],
    ("attn_bwd", "bf16"): ["bwd_sm103.cu"],
    ("attn_bwd", "f32"): ["simt_attn.cu"],
}


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libattn.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    stamp = _stamp(extra_flags)
    stamp_file = os.path.join(BUILD, "stamp")
    if (not force and os.path.exists(LIB) and os.path.exists(stamp_file)
            and open(stamp_file).read() == stamp):
        return LIB
    cc = nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs, "-lrt", "-ldl",
           "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
