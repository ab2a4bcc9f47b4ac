"""Build libpkv.so (the CUDA kernels and the C ABI) in place, for sm_103a only.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library next to this file. The CUDA runtime is linked statically, so the
library needs only the driver at run time; it builds the same way on x86_64
and aarch64 hosts.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(HERE, "libpkv.so")
SOURCES = ["kv_store.cu", "decode.cu", "prefill.cu", "api.cu", "decode_noalloc.cu",
           "block_manager.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _needs_rebuild() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    lib_time = os.path.getmtime(LIBRARY)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    include = os.path.join(ROOT, "include")
    deps += [os.path.join(include, f) for f in os.listdir(include)]
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > lib_time for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not _needs_rebuild():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        proc = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, cmd, proc

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        results = list(pool.map(compile_one, SOURCES))
    errors = []
    for src, obj, cmd, proc in results:
        if verbose or proc.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + proc.stdout + proc.stderr)
        if proc.returncode != 0:
            errors.append(src)
    if errors:
        raise RuntimeError("nvcc failed for " + ", ".join(errors))
    tmp = LIBRARY + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [r[1] for r in results]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError("link failed:\n" + proc.stdout + proc.stderr)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else []))
