"""Compile libcsa2.so (and the input generator's libcsa2_synth.so, and the tensor-rate
probe libcsa2_peak.so that bench.py uses for the FP4 roofline denominator) for sm_103a.

Each .cu is compiled to an object in parallel with nvcc, then linked into a shared
library next to its sources' package.  Run ``python -m
compressed_sparse_attention_04_gb300.build`` or call ``build_all()``.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return cand


def _compile_one(nvcc, src, obj, log_dir):
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(log_dir, os.path.basename(src) + ".ptxas.txt")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
    return obj


def _newer(out, srcs):
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(s) <= t for s in srcs)


def build_lib(src_dir, out_path, extra_deps=(), force=False):
    srcs = sorted(os.path.join(src_dir, f) for f in os.listdir(src_dir) if f.endswith(".cu"))
    deps = srcs + sorted(os.path.join(src_dir, f) for f in os.listdir(src_dir)
                         if f.endswith((".cuh", ".h"))) + list(extra_deps)
    if not force and _newer(out_path, deps):
        return out_path
    nvcc = _nvcc()
    bdir = os.path.join(os.path.dirname(out_path), "_build")
    os.makedirs(bdir, exist_ok=True)
    objs = [os.path.join(bdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        list(ex.map(lambda so: _compile_one(nvcc, so[0], so[1], bdir), zip(srcs, objs)))
    tmp = out_path + ".tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed for {out_path}:\n{r.stderr[-4000:]}")
    os.replace(tmp, out_path)
    return out_path


def build_all(force=False):
    lib = build_lib(os.path.join(PKG_DIR, "csrc"), os.path.join(PKG_DIR, "libcsa2.so"),
                    extra_deps=[os.path.join(ROOT, "include", "csa2.h")], force=force)
    syn = build_lib(os.path.join(ROOT, "synth", "csrc"), os.path.join(ROOT, "synth", "libcsa2_synth.so"),
                    force=force)
    build_lib(os.path.join(PKG_DIR, "peak"), os.path.join(PKG_DIR, "peak", "libcsa2_peak.so"), force=force)
    return lib, syn


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv))
