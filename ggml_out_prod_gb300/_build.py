"""Compile the CUDA library in-tree for sm_103a (nvcc only, no cmake).

Each translation unit compiles in parallel to an object file under
``ggml_out_prod_gb300/_build``; they link into ``liboop.so`` there.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(BUILD, "liboop.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build")
    return cand


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hdrs


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


# Host code built with AddressSanitizer and UndefinedBehaviorSanitizer (device
# code unchanged), into its own folder: for the CPU tests of the host-side
# checks, loaded with the sanitizer runtimes preloaded.
SANITIZE = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined",
            "-Xcompiler", "-fno-omit-frame-pointer", "-Xcompiler", "-fno-sanitize-recover=all"]


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          sanitize: bool = False) -> str:
    build_dir = os.path.join(BUILD, "sanitize") if sanitize else BUILD
    so = os.path.join(build_dir, "liboop.so")
    if sanitize:
        extra = list(extra or []) + SANITIZE
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    hdrs = _deps()
    objs = []
    jobs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs + [__file__]):
            cmd = [cc, *ARCH, *NVCC_FLAGS, *(extra or []), "-c", src, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(so, objs):
        tmp = so + f".{os.getpid()}.tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath,/usr/local/cuda/lib64", *(SANITIZE if sanitize else [])]
        run(cmd)
        os.replace(tmp, so)
    return so


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
