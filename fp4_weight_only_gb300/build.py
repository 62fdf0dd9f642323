"""In-tree build of the CUDA library ``_petit.so`` for sm_103a.

Each ``csrc/*.cu`` file is compiled in parallel with nvcc into ``_build/``
and linked into one shared library next to this file (CUDA runtime linked
statically; the driver API is reached through the runtime's entry-point
query, so the library loads without libcuda on a machine with no GPU).

``build_check()`` makes the bounds-checking build ``_petit_check.so`` (same
sources and API, compiled with ``-DPETIT_CHECK_BOUNDS`` into
``_build_check/``): the GEMM kernel checks every buffer index and copy
before use and reports a failed check as a status instead of faulting.
"""

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "_petit.so")
BUILD_CHECK = os.path.join(HERE, "_build_check")
CHECK_LIB = os.path.join(HERE, "_petit_check.so")
CHECK_FLAGS = ["-DPETIT_CHECK_BOUNDS"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "petit.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force=False, verbose=False, extra_flags=(), lib=LIB, build_dir=BUILD):
    """Compile and link the library if any input is newer than it."""
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            errors.append(f"{os.path.basename(src)}:\n{text}")
        elif verbose and text.strip():
            print(text, file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib)
    return lib


def build_check(force=False, verbose=False):
    """The bounds-checking build, ``_petit_check.so``."""
    return build(force, verbose, CHECK_FLAGS, CHECK_LIB, BUILD_CHECK)


if __name__ == "__main__":
    check = "--check" in sys.argv
    fn = build_check if check else build
    print(fn(force="--force" in sys.argv, verbose=True))
