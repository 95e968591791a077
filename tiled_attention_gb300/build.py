"""Build libtiled_attn.so (sm_103a) in-tree with nvcc: one object per translation unit,
compiled in parallel, then linked with the static CUDA runtime. No torch, no cmake."""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "libtiled_attn.so")
HEADER = os.path.join(ROOT, "include", "attn.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (glob.glob(os.path.join(CSRC, "*")) + [HEADER, os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every .cu under csrc/ and link the shared library; returns its path."""
    if not force and not extra_flags and up_to_date():
        return LIB
    os.makedirs(LIB_DIR, exist_ok=True)
    objs_dir = os.path.join(LIB_DIR, "obj")
    os.makedirs(objs_dir, exist_ok=True)
    nv = nvcc()

    def compile_one(src):
        obj = os.path.join(objs_dir, os.path.basename(src) + ".o")
        cmd = [nv, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, sources()))
    failed = [(s, r) for s, _, r in results if r.returncode != 0]
    if verbose:
        for s, _, r in results:
            sys.stderr.write(r.stderr)
    if failed:
        msg = "\n".join(f"== {s}\n{r.stdout}{r.stderr}" for s, r in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [nv, *ARCH, "-shared", "-o", tmp, *[o for _, o, _ in results]]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
