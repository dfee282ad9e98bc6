"""Build libgdn.so in place: every ``csrc/*.cu`` compiled for sm_103a with nvcc,
in parallel, then linked into one shared library next to this file.

With GDN_CHECKS=1 in the environment (or checks=True) the bounds-checked
variant is built instead, as libgdn_checks.so: every thread-issued global
store of the prefill and decode kernels is checked against its buffer, and a
failed check is reported by gdn_device_status as GDN_ERR_BOUNDS."""
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")

def checks_enabled() -> bool:
    return os.environ.get("GDN_CHECKS", "0") not in ("", "0")


BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgdn.so")
BUILD_CHECKS = os.path.join(HERE, "_build_checks")
LIB_CHECKS = os.path.join(HERE, "libgdn_checks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib=LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps() + [__file__])


def build(force: bool = False, verbose: bool = False, extra=(), checks=None) -> str:
    """Compile and link libgdn.so (libgdn_checks.so for the bounds-checked
    variant) unless it is newer than every source."""
    if checks is None:
        checks = checks_enabled()
    LIB, BUILD = (LIB_CHECKS, BUILD_CHECKS) if checks else (globals()["LIB"], globals()["BUILD"])
    if checks:
        extra = tuple(extra) + ("-DGDN_CHECKS",)
    if not force and up_to_date(LIB):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    cuda = os.path.dirname(os.path.dirname(nvcc)) if os.path.isabs(nvcc) else "/usr/local/cuda"
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath=" + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checks=("--checks" in sys.argv) or None))
