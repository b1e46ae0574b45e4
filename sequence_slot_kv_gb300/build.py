"""Build libslotkv.so in place for sm_103a.

The translation units compile in parallel (one per head dim for the decode
and the tensor-core prefill kernels, the host side, the allocation-free
entry point), then link into ``sequence_slot_kv_gb300/libslotkv.so``.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libslotkv.so")
OBJDIR = os.path.join(HERE, "_build")
SOURCES = ["slotkv.cu", "decode_attn_hd64.cu", "decode_attn_hd128.cu", "decode_attn_hd256.cu",
           "noalloc.cu", "prefill_tc_hd64.cu", "prefill_tc_hd128.cu"]
DEPS = ["params.h", "decode_attn.cuh", "decode_small.cuh", "prefill_tc.cuh", "tc_ops.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE] + ARCH


def _cuda_home():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _stale(out, srcs):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def build(force=False, verbose_ptxas=False):
    os.makedirs(OBJDIR, exist_ok=True)
    header = os.path.join(INCLUDE, "slotkv.h")
    deps = [os.path.join(CSRC, d) for d in DEPS] + [header]
    procs, objs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OBJDIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [path] + deps):
            cmd = ["nvcc"] + NVCC_FLAGS + ["-c", path, "-o", obj]
            if verbose_ptxas:
                cmd += ["-Xptxas", "-v"]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if verbose_ptxas or pr.returncode != 0:
            sys.stdout.write(out)
        if pr.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if force or _stale(LIB, objs):
        cuda_lib = os.path.join(_cuda_home(), "lib64")
        cmd = ["nvcc", "-shared", "-o", LIB] + objs + ARCH + [
            "-cudart", "shared", "-Xlinker", "-rpath=" + cuda_lib]
        subprocess.run(cmd, check=True)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
