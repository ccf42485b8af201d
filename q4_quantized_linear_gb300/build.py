"""Build libq4mm.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit compiles in parallel; the shared object links the
CUDA runtime statically and exports only the q4_* C ABI.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libq4mm.so")
TRACE_BUILD = os.path.join(PKG, "_build_trace")
TRACE_LIB = os.path.join(TRACE_BUILD, "libq4mm.so")
CHECKED_BUILD = os.path.join(PKG, "_build_checked")
CHECKED_LIB = os.path.join(CHECKED_BUILD, "libq4mm.so")
HEADER = os.path.join(ROOT, "include", "q4mm.h")

SOURCES = ["q4mm_api.cu", "q4mm_pack.cu", "q4mm_decode.cu", "q4mm_gemv.cu", "q4mm_mmv.cu", "q4mm_matvec.cu", "q4mm_w8.cu", "q4mm_prefill.cu",
           "q4mm_static.cu", "q4mm_gguf.cu", "q4mm_experts.cu"]
DEPS = ["q4mm_device.cuh", "q4mm_internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libq4mm")
    return path


def _stale(target: str, inputs: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def _compile(src: str, verbose_ptxas: bool, outdir: str = BUILD, extra: tuple = ()) -> str:
    obj = os.path.join(outdir, os.path.splitext(src)[0] + ".o")
    inputs = [os.path.join(CSRC, src), HEADER] + [os.path.join(CSRC, d) for d in DEPS] + [__file__]
    if not _stale(obj, inputs):
        return obj
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + list(extra) + (["-Xptxas", "-v"] if verbose_ptxas else []) + \
        ["-c", os.path.join(CSRC, src), "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas and r.stderr:
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, trace: bool = False, checked: bool = False) -> str:
    """Compile libq4mm. trace=True makes the profiling build (in-kernel event
    trace, -DQ4MM_TRACE), checked=True the debug build whose decode kernel
    checks its indices and offsets and reports a failed check in the status
    word (-DQ4MM_CHECKED); each in a directory of its own."""
    if trace:
        outdir, lib, extra = TRACE_BUILD, TRACE_LIB, ("-DQ4MM_TRACE",)
    elif checked:
        outdir, lib, extra = CHECKED_BUILD, CHECKED_LIB, ("-DQ4MM_CHECKED",)
    else:
        outdir, lib, extra = BUILD, LIB, ()
    os.makedirs(outdir, exist_ok=True)
    if force:
        for f in os.listdir(outdir):
            if f.endswith(".o"):
                os.remove(os.path.join(outdir, f))
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, outdir, extra), SOURCES))
    if force or _stale(lib, objs):
        vscript = os.path.join(outdir, "exports.map")
        with open(vscript, "w") as f:
            f.write("{ global: q4_*; local: *; };\n")
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + \
            ["-Xlinker", f"--version-script={vscript}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, trace="--trace" in sys.argv,
                checked="--checked" in sys.argv))
