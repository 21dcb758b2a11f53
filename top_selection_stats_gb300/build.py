"""Build libsmp.so (the CUDA library behind include/smp.h) in-tree for sm_103a.

The host API and the three element-type instantiations of the kernel are
separate translation units, compiled in parallel and linked into one shared
library.
"""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libsmp.so")
OBJDIR = os.path.join(HERE, "_build")
SOURCES = [os.path.join(CSRC, f) for f in ("smp_api.cu", "smp_k_f32.cu", "smp_k_bf16.cu",
                                           "smp_k_f16.cu", "smp_verify.cu", "smp_penalty.cu",
                                           "smp_gumbel.cu", "smp_toplp.cu", "smp_x_bf16.cu",
                                           "smp_x_f16.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("smp_philox.cuh", "smp_device.cuh", "smp_core.cuh",
                                           "smp_list.cuh",
                                           "smp_stream_passes.cuh", "smp_general.cuh",
                                           "smp_kernel.cuh", "smp_split.cuh")]
DEPS = SOURCES + HEADERS + [os.path.join(ROOT, "include", "smp.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr"]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def _run(cmd):
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    return res.stdout + res.stderr


def build(force=False, verbose=False, extra=()):
    """Compile the library unless it is newer than every source."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    objs, cmds = [], []
    for src in SOURCES:
        obj = os.path.join(OBJDIR, os.path.basename(src) + ".o")
        objs.append(obj)
        cmds.append([nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj])
    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        logs = list(ex.map(_run, cmds))
    tmp = LIB + ".tmp"
    logs.append(_run([nvcc(), *ARCH, "-shared", *objs, "-o", tmp]))
    if verbose:
        print("".join(logs))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True, extra=("-Xptxas", "-v")))
