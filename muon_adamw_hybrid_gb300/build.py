"""In-tree build of the CUDA libraries with nvcc for sm_103a.

    python muon_adamw_hybrid_gb300/build.py      (or __graft_entry__.build())

compiles every translation unit in parallel and links

    muon_adamw_hybrid_gb300/libmuonhybrid.so   (the optimizer step, C ABI)
    synth/libmhsynth.so                        (seeded input generator)

Both link the CUDA runtime statically and use no other CUDA library, so the
only run-time requirement is the driver.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]

LIBS = {
    os.path.join(PKG, "libmuonhybrid.so"): [
        os.path.join(CSRC, f) for f in ("api.cu", "adamw.cu", "elementwise.cu", "ns_gemm.cu",
                                             "noalloc.cu", "grad_control.cu", "qk_clip.cu")
    ],
    os.path.join(ROOT, "synth", "libmhsynth.so"): [os.path.join(ROOT, "synth", "synth.cu")],
}


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")
    return path


def _run(cmd):
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    return res.stdout + res.stderr


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra_flags=()) -> list[str]:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    jobs = []
    objs = {}
    for lib, srcs in LIBS.items():
        objs[lib] = []
        for src in srcs:
            obj = os.path.join(BUILD, os.path.basename(src) + ".o")
            objs[lib].append(obj)
            if force or _stale(obj, [src] + headers):
                jobs.append([nvcc(), *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj])
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for out in ex.map(_run, jobs):
            if verbose and out.strip():
                print(out)
    built = []
    for lib, ob in objs.items():
        if force or _stale(lib, ob):
            tmp = lib + ".tmp"
            _run([nvcc(), *ARCH, "-shared", "-o", tmp, *ob])
            os.replace(tmp, lib)
        built.append(lib)
    return built


if __name__ == "__main__":
    extra = [a for a in sys.argv[1:] if a.startswith("-X") or a.startswith("--")]
    for p in build(verbose=True, force="--force" in sys.argv,
                   extra_flags=[a for a in extra if a != "--force"]):
        print(p)
