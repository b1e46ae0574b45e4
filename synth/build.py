"""Build the synthetic-input generator libraries in place.

``libsynth_host.so`` (gcc) fills host arrays; ``libsynth_dev.so`` (nvcc,
sm_103a) fills device buffers with the same values.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libsynth_host.so")
DEV_LIB = os.path.join(HERE, "libsynth_dev.so")


def _stale(out, srcs):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def host_cmd():
    src = os.path.join(HERE, "synth_host.c")
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-Wall", "-Wextra", "-o", HOST_LIB, src, "-lpthread"]


def dev_cmd():
    src = os.path.join(HERE, "synth_dev.cu")
    return ["nvcc", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
            "-o", DEV_LIB, src]


def build_host(force=False):
    srcs = [os.path.join(HERE, f) for f in ("synth_host.c", "synth.h")]
    if force or _stale(HOST_LIB, srcs):
        subprocess.run(host_cmd(), check=True)
    return HOST_LIB


def build_dev(force=False):
    srcs = [os.path.join(HERE, f) for f in ("synth_dev.cu", "synth.h")]
    if force or _stale(DEV_LIB, srcs):
        subprocess.run(dev_cmd(), check=True)
    return DEV_LIB
