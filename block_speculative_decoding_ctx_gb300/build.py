"""Build libdflash.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel to an object in
_build/, then linked into block_speculative_decoding_ctx_gb300/libdflash.so.
A unit is recompiled when it, or any header it may include, is newer than its
object.  No cmake, no torch extension machinery.
"""

import concurrent.futures
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdflash.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(src, obj, hdr_mtime):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or hdr_mtime > t


def build(verbose=False, extra_flags=()):
    """Compile what is stale and link.  DFLASH_NVCC_FLAGS (environment) adds
    compile flags, e.g. -D defaults of the launch heuristics."""
    extra_flags = tuple(extra_flags) + tuple(os.environ.get("DFLASH_NVCC_FLAGS", "").split())
    os.makedirs(BUILD, exist_ok=True)
    # the GEMM instantiation units take longest: start them first
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")),
                  key=lambda p: (not os.path.basename(p).startswith("gemm_tiles"), -os.path.getsize(p), p))
    hdr_mtime = max([os.path.getmtime(h) for h in _headers()] + [0.0])
    cc = nvcc()
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        if _stale(src, obj, hdr_mtime):
            jobs.append([cc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj])
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for err in ex.map(run, jobs):
            if verbose and err:
                print(err, file=sys.stderr)
    need_link = bool(jobs) or not os.path.exists(LIB) or \
        any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs)
    if need_link:
        run([cc, *ARCH, "-shared", "-o", LIB + ".tmp", *objs, "-lcudart_static", "-ldl", "-lrt",
             "-lpthread"])
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
