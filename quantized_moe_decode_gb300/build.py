"""Build libuocr.so in-tree with nvcc for sm_103a (parallel compile, one link).

    python -m quantized_moe_decode_gb300.build [--force] [--ptxas-v] [--out PATH] [-DNAME=VALUE ...]

The library is rebuilt when any source under csrc/ or include/ is newer than
it.  Objects go to quantized_moe_decode_gb300/_build/ (a subfolder per --out
target).  -D defines select the build-time tuning of csrc/device_common.cuh
(UOCR_RING_DEPTH, UOCR_MIN_BLOCKS, UOCR_UNROLL); a variant built with --out
is loaded by pointing UOCR_LIB at it.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libuocr.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra, bdir: str = BUILD):
    obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, extra=(), out: str = LIB) -> str:
    """Compile every .cu under csrc/ and link libuocr.so (or `out`); returns its path."""
    if not force and not _stale(out):
        return out
    bdir = BUILD if out == LIB else os.path.join(BUILD, os.path.basename(out).replace(".", "_"))
    os.makedirs(bdir, exist_ok=True)
    srcs = sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        done = list(ex.map(lambda s: _compile(s, list(extra), bdir), srcs))
    objs = [o for o, _ in done]
    if verbose:
        for _, log in done:
            if log:
                print(log, end="")
    tmp = out + ".tmp"
    cmd = [NVCC, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(f"built {out}")
    return out


if __name__ == "__main__":
    argv = sys.argv[1:]
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in argv else []
    extra += [a for a in argv if a.startswith("-D")]
    out = os.path.abspath(argv[argv.index("--out") + 1]) if "--out" in argv else LIB
    build(force="--force" in argv or out != LIB, verbose=True, extra=extra, out=out)
