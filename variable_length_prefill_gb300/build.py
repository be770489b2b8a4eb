"""Build the CUDA library in-tree with nvcc for sm_103a.

Produces ``variable_length_prefill_gb300/_lib/libattn_varlen.so`` from the
sources in ``csrc/``.  Each translation unit compiles in its own nvcc
process, in parallel; the link step uses the static CUDA runtime so the
library needs only the driver at run time.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "libattn_varlen.so"
# Test-only builds: the same sources with extra defines, in a library of their
# own that the product never loads.  "testhooks" shortens every kernel wait to
# 50 ms and compiles the hook that withholds one K/V tile, so a test can run
# a wait out and check the reported status.
VARIANTS = {
    "testhooks": ("libattn_varlen_testhooks.so",
                 ["-DATTN_VARLEN_WAIT_LIMIT_NS=50000000ull", "-DATTN_VARLEN_TEST_HOOKS=1"]),
}
SOURCES = ["attn_varlen_api.cu", "attn_varlen_kernels.cu", "attn_varlen_d256.cu",
           "paged_decode.cu", "chunk_o.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-I", INCLUDE, "-I", CSRC]


def lib_path(variant: str | None = None) -> str:
    name = LIB_NAME if variant is None else VARIANTS[variant][0]
    return os.path.join(LIB_DIR, name)


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _fingerprint(extra: list) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, variant: str | None = None) -> str:
    """Compile (if sources changed) and return the library path.

    ``variant``: a key of VARIANTS to build that test-only library instead."""
    os.makedirs(LIB_DIR, exist_ok=True)
    out = lib_path(variant)
    extra = [] if variant is None else VARIANTS[variant][1]
    stamp = out + ".sha256"
    fp = _fingerprint(extra)
    if not force and os.path.exists(out) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == fp:
                return out
    nvcc = _nvcc()
    objs, procs = [], []
    tag = "" if variant is None else "_" + variant
    for src in SOURCES:
        obj = os.path.join(LIB_DIR, src.replace(".cu", f"{tag}.o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
    failed = []
    for cmd, p in procs:
        log, _ = p.communicate()
        if verbose and log:
            print(log)
        if p.returncode != 0:
            failed.append((" ".join(cmd), log))
    if failed:
        msg = "\n\n".join(f"$ {c}\n{log}" for c, log in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = out + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n$ {' '.join(link)}\n{r.stdout}{r.stderr}")
    os.replace(tmp, out)
    for obj in objs:
        os.remove(obj)
    with open(stamp, "w") as f:
        f.write(fp)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
