"""Build libfa.so in-tree with nvcc for sm_103a (one -gencode, parallel TUs).

    python -m exact_attention_44_gb300.build [--force] [--verbose] [--debug-checks]

Objects and the shared library go to exact_attention_44_gb300/_build/ (git
ignored).  A content hash of the sources, headers and flags is stored next to
the library; an unchanged tree is not rebuilt.  --debug-checks builds a
second library, _build/checks/libfa.so, whose forward kernels check every
unit they decode against the launch's sizes (FA_DEBUG_CHECKS=1).
"""
from __future__ import annotations

import argparse
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libfa.so")

# (source, object, extra flags): the per-head-dim launchers are one source
# each, compiled once per supported head dim
FWD_DIMS = (16, 32, 64, 128, 256)
BWD_DIMS = (16, 32, 64, 128, 256)
UNITS = ([(src, src.replace(".cu", ".o"), []) for src in ("fa_api.cu", "fa_lse_merge.cu", "fa_noalloc.cu")] +
         [("fa_fwd_dim.cu", f"fa_fwd_d{d}.o", [f"-DFA_HEAD_DIM={d}"]) for d in FWD_DIMS] +
         [("fa_bwd_dim.cu", f"fa_bwd_d{d}.o", [f"-DFA_HEAD_DIM={d}"]) for d in BWD_DIMS])
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libfa needs the CUDA 13 toolkit to build")


def _tree_hash(extra_flags: list[str]) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode() + b"\0" + f.read())
    h.update(" ".join(FLAGS + extra_flags).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug_checks: bool = False) -> str:
    """Compile every translation unit (in parallel) and link libfa.so; returns its path.

    debug_checks: build the index-checking variant into _build/checks/ instead."""
    extra_flags = list(extra_flags or [])
    build_dir, lib_path = BUILD, LIB
    if debug_checks:
        extra_flags.append("-DFA_DEBUG_CHECKS=1")
        build_dir = os.path.join(BUILD, "checks")
        lib_path = os.path.join(build_dir, "libfa.so")
    os.makedirs(build_dir, exist_ok=True)
    digest = _tree_hash(extra_flags)
    stamp = lib_path + ".hash"
    if not force and os.path.exists(lib_path) and os.path.exists(stamp) and open(stamp).read() == digest:
        return lib_path
    cc = nvcc()
    jobs = []
    for src, obj_name, unit_flags in UNITS:
        obj = os.path.join(build_dir, obj_name)
        cmd = [cc, *FLAGS, *unit_flags, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((src, obj, cmd))

    def run(job):
        src, obj, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return os.path.basename(obj), r

    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(run, jobs))
    failed = False
    for src, r in results:
        if r.returncode != 0:
            failed = True
            sys.stderr.write(f"--- nvcc failed on {src}\n{r.stdout}{r.stderr}\n")
        elif verbose and (r.stdout or r.stderr):
            sys.stderr.write(f"--- {src}\n{r.stdout}{r.stderr}\n")
    if failed:
        raise RuntimeError("libfa build failed")
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [cc, *ARCH, "-shared", "-o", tmp, *[obj for _, obj, _ in jobs]]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"libfa link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib_path


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/spill/smem usage")
    ap.add_argument("--debug-checks", action="store_true",
                    help="build the variant whose kernels check every unit against the launch's sizes")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, debug_checks=a.debug_checks))


if __name__ == "__main__":
    main()
