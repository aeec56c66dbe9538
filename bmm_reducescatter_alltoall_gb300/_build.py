"""Build libbmmrsa2a.so in-tree with nvcc for sm_103a.

Each translation unit in csrc/ is compiled in parallel to an object under
_build/, then linked into lib/libbmmrsa2a.so (CUDA runtime linked
statically, so the library loads without a GPU driver present).  A stamp
file holding a hash of the sources and flags skips the work when nothing
changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libbmmrsa2a.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
          "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbmmrsa2a.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sorted(hs)


def _digest(extra) -> str:
    h = hashlib.sha256()
    for p in _sources() + _headers():
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + CFLAGS + list(extra)).encode())
    return h.hexdigest()


KERNEL_SOURCES = {
    "fused_tc_kernel": "fused_tc.cu",
    "fused_tc2_kernel": "fused_tc2.cu",
    "fused_tcu_kernel": "fused_tcu.cu",
    "fused_tcr_kernel": "fused_tcr.cu",
    "l2_flush_kernel": "l2_flush.cu",
    "fused_simt_kernel": "fused_simt.cu",
    "a2av_kernel": "a2av.cu",
    "ia2av_kernel": "ia2av.cu",
    "repack_rows_kernel": "repack.cu",
    "mma_probe_kernel": "mma_probe.cu",
    "gather_probe_kernel": "gather_probe.cu",
}


def code_text(src: bytes) -> bytes:
    """C/C++/CUDA source with comments removed and whitespace normalised
    (runs of blanks become one space, blank lines dropped); string and
    character literals are kept verbatim.  Two sources with the same code
    text compile to the same program."""
    out = bytearray()
    i, n = 0, len(src)
    while i < n:
        c = src[i:i + 1]
        if c == b"/" and src[i + 1:i + 2] == b"/":
            j = src.find(b"\n", i)
            i = n if j < 0 else j
        elif c == b"/" and src[i + 1:i + 2] == b"*":
            j = src.find(b"*/", i + 2)
            i = n if j < 0 else j + 2
            out += b" "
        elif c in (b'"', b"'"):
            j = i + 1
            while j < n and src[j:j + 1] != c:
                j += 2 if src[j:j + 1] == b"\\" else 1
            out += src[i:j + 1]
            i = j + 1
        else:
            out += c
            i += 1
    lines = (b" ".join(line.split()) for line in bytes(out).split(b"\n"))
    return b"\n".join(line for line in lines if line)


def included_files(path: str) -> list:
    """`path` and every header it includes with #include "..." (found in
    csrc/ or include/), transitively, each once, in a stable order."""
    seen, order = set(), []

    def visit(p):
        if p in seen:
            return
        seen.add(p)
        order.append(p)
        with open(p, "rb") as f:
            text = code_text(f.read()).decode("utf-8", "replace")
        for line in text.splitlines():
            line = line.strip()
            if line.startswith("#include") and '"' in line:
                name = line.split('"')[1]
                for d in (os.path.dirname(p), CSRC, INCLUDE):
                    q = os.path.join(d, name)
                    if os.path.exists(q):
                        visit(os.path.normpath(q))
                        break
    visit(os.path.normpath(path))
    return order


def source_digest(kernel: str = None) -> str:
    """Hash identifying a kernel build: the code text (comments and
    whitespace ignored) of the kernel's translation unit and of the headers
    it includes, and the compile flags (all sources, verbatim, when `kernel`
    is None)."""
    if kernel is None:
        return _digest([])
    h = hashlib.sha256()
    for p in included_files(os.path.join(CSRC, KERNEL_SOURCES[kernel])):
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(code_text(f.read()))
    h.update(" ".join(ARCH + CFLAGS).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link; returns the library path."""
    extra = list(extra_flags)
    stamp = os.path.join(BUILD_DIR, "stamp")
    digest = _digest(extra)
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = _nvcc()
    # The visible declarations of the public header carry default visibility.
    defs = ["-DBRA_BUILD"]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *CFLAGS, *defs, *extra, "-I", INCLUDE, "-I", CSRC,
               "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
