"""Build libmsa.so (the MSA C-ABI library) in-tree for sm_103a with nvcc.

Usage: python -m segmented_kv_attention_msa_b300.build [-v] [--debug]

--debug builds libmsa_debug.so instead: the same library compiled with MSA_DEBUG, whose
kernels check every work record, block id and block fill they read against the plan and
the pool, record MSA_ERR_BLOCK_OOB in the status word and substitute a safe value instead
of trapping.  The package loads it when MSA_LIBRARY=debug is set in the environment.
"""
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmsa.so")
DEBUG_LIB = os.path.join(PKG, "libmsa_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(f) > t for f in deps)


def build(verbose: bool = False, force: bool = False, extra=(), debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    if not force and not needs_build(lib):
        return lib
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
           "-Xcompiler", "-fPIC", "-shared", "-I" + INCLUDE, "-I" + CSRC,
           "-Xptxas", "-v" if verbose else "-O3", *(["-DMSA_DEBUG"] if debug else []), *extra,
           "-o", lib + ".tmp", *sources()]
    if verbose:
        print(" ".join(cmd))
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force=True, debug="--debug" in sys.argv))
