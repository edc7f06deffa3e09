"""Build libspx.so (sm_103a) in-tree with nvcc.

Each .cu file is compiled to an object in parallel, then linked into a shared
library against the shared CUDA runtime (so the process keeps a single
runtime instance alongside PyTorch).  Output: ``_build/libspx.so``.

``build(variant="timeline")`` builds the profiling library
``_build/timeline/libspx_timeline.so`` instead: the same sources with
``-DSPX_TIMELINE``, whose draft launch records %globaltimer phase marks
(``spx_timeline_reset`` / ``spx_timeline_read``).  The product never loads it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libspx.so")
VARIANTS = {None: (BUILD, LIB, []),
            "timeline": (os.path.join(BUILD, "timeline"), os.path.join(BUILD, "timeline", "libspx_timeline.so"),
                         ["-DSPX_TIMELINE"])}
SOURCES = ["spx_route.cu", "spx_engine.cu", "spx_draft.cu", "spx_pack.cu", "spx_api.cu", "spx_noalloc.cu",
           "spx_plan.cu", "spx_tc.cu"]
# every header of csrc/ and the public one: a change to any rebuilds every source
HEADERS = sorted(f for f in os.listdir(CSRC) if f.endswith(".cuh")) + [os.path.join("..", "..", "include", "spx.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspx")
    return p


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, variant: str | None = None) -> str:
    bdir, lib, extra = VARIANTS[variant]
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS]
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + hdrs):
            cmd = [cc, *ARCH, *FLAGS, *extra, "-c", s, "-o", o]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append((src, cmd))
    objs = [os.path.join(bdir, s.replace(".cu", ".o")) for s in SOURCES]

    def run(job):
        name, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return name, r.returncode, r.stdout + r.stderr

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for name, rc, out in ex.map(run, jobs):
                if verbose or rc != 0 or ptxas_info:
                    sys.stderr.write(out)
                if rc != 0:
                    raise RuntimeError(f"nvcc failed on {name}")
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart=shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link of libspx.so failed")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                variant="timeline" if "--timeline" in sys.argv else None))
