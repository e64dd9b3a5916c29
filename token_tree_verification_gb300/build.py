"""Build ``libspec_tree.so`` in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` file is compiled in parallel to an object under ``_build/``
and linked into one shared library next to this file.  The CUDA runtime is
linked statically, so the library needs only the driver at run time.

``build(checked=True)`` makes the bounds-checked debug build instead
(``-DSPEC_CHECKED``, objects under ``_build/spec_tree_checked``, output
``libspec_tree_checked.so``); ``binding.load()`` opens it when the
environment sets ``SPEC_TREE_CHECKED=1``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libspec_tree.so")
BUILD_DIR = os.path.join(os.path.dirname(HERE), "_build", "spec_tree")
OUT_CHECKED = os.path.join(HERE, "libspec_tree_checked.so")
BUILD_DIR_CHECKED = os.path.join(os.path.dirname(HERE), "_build", "spec_tree_checked")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers() -> list[str]:
    inc = os.path.join(os.path.dirname(HERE), "include")
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return hs


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    build_dir = BUILD_DIR_CHECKED if checked else BUILD_DIR
    out = OUT_CHECKED if checked else OUT
    flags = FLAGS + (["-DSPEC_CHECKED"] if checked else [])
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = sources()
    hdrs = _headers()
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(src, obj):
        if force or _stale(obj, [src] + hdrs):
            cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose:
                print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        list(ex.map(lambda p: compile_one(*p), zip(srcs, objs)))
    if force or _stale(out, objs):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
