"""Builds libmoe_gb300.so in-tree from csrc/*.cu for sm_103a.

Each translation unit is compiled in parallel with nvcc, then linked into a
shared library (CUDA runtime linked statically, no driver library needed at
link time: the tensor-map encoder is looked up at run time).
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libmoe_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
# Debug build: the same sources with -DMOE_DEBUG (index, segment and TMA
# coordinate checks that record MOE_ERR_ARG instead of touching memory
# outside a buffer); used by the tests, never by the benchmark.
DEBUG_OUT_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_OUT_DIR, LIB_NAME)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-diag-suppress", "1160"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _code_only(text: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace collapsed
    (string literals kept as they are)."""
    import re
    token = re.compile(r'"(?:\\.|[^"\\])*"|//[^\n]*|/\*.*?\*/', re.S)
    code = token.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return " ".join(code.split())


def source_digest(root: str = None) -> str:
    """First 16 hex digits of a SHA-256 over the code (comments and
    whitespace aside) of the library's CUDA/C++ sources and its public
    header: names a build of the kernels, so a profile taken of one build is
    not read as a measurement of another.  `root`: a directory holding
    csrc/ and include/moe.h laid out as in the repository (default: this
    package)."""
    import hashlib
    csrc = os.path.join(root, "csrc") if root else CSRC
    header = os.path.join(root, "include", "moe.h") if root else os.path.join(HERE, "..", "include", "moe.h")
    h = hashlib.sha256()
    names = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in names:
        h.update(f.encode())
        h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    h.update(_code_only(open(header, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def build(verbose: bool = False, debug: bool = False) -> str:
    out_dir, lib_path = (DEBUG_OUT_DIR, DEBUG_LIB_PATH) if debug else (OUT_DIR, LIB_PATH)
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = sources()
    objs = [os.path.join(out_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    flags = FLAGS + (["-DMOE_DEBUG"] if debug else [])

    def compile_one(pair):
        src, obj = pair
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r.returncode, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, zip(srcs, objs)))
    failed = [(s, log) for s, rc, log in results if rc != 0]
    for s, rc, log in results:
        if verbose or rc != 0:
            sys.stderr.write(f"== {os.path.basename(s)} ==\n{log}\n")
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(s) for s, _ in failed))
    tmp = lib_path + ".tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, debug="--debug" in sys.argv))
