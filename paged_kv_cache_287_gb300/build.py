"""Build libpagedattn.so in-tree with nvcc for sm_103a (GB300).

Translation units compile in parallel; the shared library links against the
shared CUDA runtime so it uses the same runtime instance as PyTorch.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedattn.so")
SOURCES = ["pa_api.cu", "pa_cache_write.cu", "pa_attention.cu",
           "pa_decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(debug: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC, "--expt-relaxed-constexpr",
                "-Xptxas", "-warn-spills"]
    if debug:
        f += ["-DPA_DEBUG=1"]
    return f


def build(verbose: bool = False, debug: bool = False, ptxas_info: bool = False,
          defines=(), out: str = LIB, build_dir: str = BUILD) -> str:
    """Compile every translation unit and link the library (default
    ``libpagedattn.so`` in the package); returns its path.  ``defines`` are
    extra ``NAME=VALUE`` preprocessor definitions (kernel tuning parameters)."""
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = _flags(debug) + (["-Xptxas", "-v"] if ptxas_info else []) + \
        [f"-D{d}" for d in defines]

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            if err.strip():
                sys.stderr.write(err)
    objs = [o for o, _ in results]
    tmp = out + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
