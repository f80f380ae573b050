"""Builds the CUDA library libgdr.so in-tree (channelwise_gated_delta_gb300/_lib/).

Every translation unit under csrc/ is compiled for sm_103a only, in parallel,
then linked into one shared library with the CUDA runtime linked statically.
The test-only diagnostics under csrc_diag/ (tensor-core operand layouts) are
linked into a separate libgdr_diag.so that the product library never loads.
Run as a script or call ``build()``.
"""
import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
CSRC_DIAG = os.path.join(HERE, "csrc_diag")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(HERE, "_lib")
# objects and the library are per host architecture: a tree copied from an
# x86_64 machine to an aarch64 one must not reuse the other's binaries
OBJ_DIR = os.path.join(ROOT, "_build", "obj-" + platform.machine())
LIB = os.path.join(LIB_DIR, "libgdr.so")
DIAG_LIB = os.path.join(LIB_DIR, "libgdr_diag.so")
STAMP = LIB + ".arch"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I" + INCLUDE, "-I" + CSRC, "--expt-relaxed-constexpr"]


def _nvcc():
    path = shutil.which("nvcc")
    if path is None and os.path.exists("/usr/local/cuda/bin/nvcc"):
        path = "/usr/local/cuda/bin/nvcc"
    if path is None:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdr.so")
    return path


def _sources(d=CSRC):
    return sorted(os.path.join(d, f) for f in os.listdir(d) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _up_to_date(target, deps):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def _compile(src, verbose, ptxas_verbose):
    obj = os.path.join(OBJ_DIR, os.path.basename(os.path.dirname(src)) + "_" +
                       os.path.basename(src) + ".o")
    if _up_to_date(obj, [src] + _headers() + [__file__]):
        return obj, ""
    cmd = [_nvcc()] + NVCC_FLAGS + (["-Xptxas", "-v"] if ptxas_verbose else []) + [
        "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return obj, r.stderr


def build(verbose=False, ptxas_verbose=False, jobs=None):
    """Compiles csrc/*.cu and links _lib/libgdr.so. Returns the library path."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = _sources()
    diag_srcs = _sources(CSRC_DIAG)
    jobs = jobs or min(len(srcs) + len(diag_srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose, ptxas_verbose), srcs + diag_srcs))
    objs = [o for o, _ in results[:len(srcs)]]
    diag_objs = [o for o, _ in results[len(srcs):]]
    if ptxas_verbose:
        for _, log in results:
            if log:
                print(log, file=sys.stderr)
    stamp_ok = os.path.exists(STAMP) and open(STAMP).read().strip() == platform.machine()
    for lib, lib_objs in ((LIB, objs), (DIAG_LIB, diag_objs)):
        if stamp_ok and _up_to_date(lib, lib_objs):
            continue
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = [_nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + lib_objs
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
        os.replace(tmp, lib)
    with open(STAMP, "w") as f:
        f.write(platform.machine() + "\n")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
