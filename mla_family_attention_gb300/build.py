"""Build the library for sm_103a: each .cu compiled by nvcc in parallel, then
linked into one shared library inside the package (in-tree, git-ignored).

    python -m mla_family_attention_gb300.build [--verbose] [--checks]

--checks builds the bounds-checked debug variant instead (-DMLA_CHECKS:
every kernel's own index and offset checks record MLA_ERR_CHECK in the
device status; nothing traps), as _build_checks/libmla_gb300_checks.so.
Set MLA_GB300_LIB to a library's path to load it in place of the default.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libmla_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
CHECKS_DIR = os.path.join(HERE, "_build_checks")
CHECKS_LIB_PATH = os.path.join(CHECKS_DIR, "libmla_gb300_checks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the library needs the CUDA 13 toolkit")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(os.path.dirname(HERE), "include", "mla.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    out_dir, lib_path = (CHECKS_DIR, CHECKS_LIB_PATH) if checks else (OUT_DIR, LIB_PATH)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _deps_mtime():
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []
    if checks:
        extra.append("-DMLA_CHECKS")
    # extra nvcc flags (e.g. -D overrides of tile or stage counts for a sweep)
    extra += os.environ.get("MLA_NVCC_FLAGS", "").split()

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv, checks="--checks" in sys.argv))
