"""Build libeqmp.so in-tree for sm_103a (no torch extension machinery).

Steps: generate the constexpr CG/SH header from csrc/gen_tables.py, compile
each translation unit with nvcc in parallel, link one shared library with
the CUDA runtime linked statically.  Output: _build/libeqmp.so next to this
file.  Re-running skips up-to-date objects.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(BUILD, "libeqmp.so")
UNITS = ["abi.cu", "shared_f32.cu", "shared_bf16.cu", "radial.cu", "bwd.cu", "so2.cu", "graph.cu", "shared_dx.cu", "hl.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _flags(verbose_ptxas=False):
    f = ["-O3", "-std=c++17", "--expt-relaxed-constexpr", "-lineinfo", "-Xcompiler", "-fPIC",
         "-I", INCLUDE, "-I", CSRC, "-I", BUILD] + ARCH
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _newest_input_mtime():
    paths = [os.path.join(CSRC, p) for p in os.listdir(CSRC)] + [os.path.join(INCLUDE, "eqmp.h")]
    return max(os.path.getmtime(p) for p in paths)


def generate_tables():
    os.makedirs(BUILD, exist_ok=True)
    out = os.path.join(BUILD, "eqmp_tables.h")
    subprocess.check_call([sys.executable, os.path.join(CSRC, "gen_tables.py"), out])
    subprocess.check_call([sys.executable, os.path.join(CSRC, "gen_tables.py"), "--high",
                           os.path.join(BUILD, "eqmp_tables_hl.h")])
    return out


def build(force=False, verbose_ptxas=False, jobs=None, out_dir=None, defines=()):
    """Compile libeqmp.so; returns its path.

    out_dir / defines build a variant elsewhere (e.g. with EQMP_TUNE_* macros
    for tuning experiments); the default is the in-tree _build/libeqmp.so.
    """
    bdir = out_dir or BUILD
    lib = os.path.join(bdir, "libeqmp.so")
    os.makedirs(bdir, exist_ok=True)
    newest = _newest_input_mtime()
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= newest and not verbose_ptxas:
        return lib
    generate_tables()
    cc = nvcc()
    dflags = [f"-D{d}" for d in defines]

    def compile_one(unit):
        obj = os.path.join(bdir, unit.replace(".cu", ".o"))
        cmd = [cc, "-c", os.path.join(CSRC, unit), "-o", obj] + _flags(verbose_ptxas) + dflags
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    with ThreadPoolExecutor(max_workers=jobs or len(UNITS)) as ex:
        results = list(ex.map(compile_one, UNITS))
    if verbose_ptxas:
        for _, err in results:
            sys.stderr.write(err)
    objs = [o for o, _ in results]
    tmp = lib + ".tmp"
    subprocess.check_call([cc, "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
