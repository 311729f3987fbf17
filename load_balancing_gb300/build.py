"""Builds libdbsp.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into
``load_balancing_gb300/libdbsp.so`` with the static CUDA runtime (so the library
loads without a GPU or a driver; the driver is opened lazily on the first CUDA
call). The tensor-map encoder is fetched through the runtime's driver entry
point, so nothing links against libcuda.
"""

import concurrent.futures
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libdbsp.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdbsp.so")


def library_path():
    return os.path.join(PKG, LIB_NAME)


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [
        os.path.abspath(__file__)]


def needs_build():
    lib = library_path()
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src, verbose, out_dir=BUILD_DIR, extra=()):
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stderr


def build(verbose=False):
    """Compile every csrc/*.cu for sm_103a and link libdbsp.so. Returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), srcs))
    objs = [o for o, _ in results]
    tmp = library_path() + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, library_path())
    if verbose:
        for _, log in results:
            if log:
                print(log)
    return library_path()


WAIT_TEST_LIB = os.path.join(BUILD_DIR, "wait_test", "libdbsp_waittest.so")


def build_wait_test():
    """Test-only library: every source compiled with -DDBSP_WAIT_TEST.

    In that build every pipeline wait of the attention kernel gives up after 20 ms,
    and the V producer of CTA 0 leaves out its first tile (neither its arrival nor its
    copy is issued), so that a wait runs out and the abort / drain / TMEM-free teardown
    runs. Likewise the streaming mask-loads kernel: 20 ms stage waits, and CTA (0, 0)
    leaves out its first stage. The product library never contains this code. Returns
    the path of the .so (under _build/).
    """
    out_dir = os.path.dirname(WAIT_TEST_LIB)
    os.makedirs(out_dir, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = [o for o, _ in ex.map(lambda s: _compile(s, False, out_dir, ["-DDBSP_WAIT_TEST"]), srcs)]
    tmp = WAIT_TEST_LIB + ".tmp"
    res = subprocess.run([nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs,
                         capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed (wait test):\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, WAIT_TEST_LIB)
    return WAIT_TEST_LIB


if __name__ == "__main__":
    import sys

    print(build(verbose="-v" in sys.argv))
