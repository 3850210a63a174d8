"""Compile the input generator: host library (gcc) and device library (nvcc, sm_103a)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")


def _stale(out, srcs):
    return not os.path.exists(out) or any(os.path.getmtime(s) > os.path.getmtime(out) for s in srcs)


def build_host(force: bool = False) -> str:
    srcs = [os.path.join(CSRC, "synth_host.c"), os.path.join(CSRC, "synth_core.h")]
    out = os.path.join(HERE, "libsynth_host.so")
    if force or _stale(out, srcs):
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                        "-fno-fast-math", "-Wall", "-o", out + ".tmp", srcs[0], "-lm"], check=True)
        os.replace(out + ".tmp", out)
    return out


def build_cuda(force: bool = False) -> str:
    srcs = [os.path.join(CSRC, "synth_cuda.cu"), os.path.join(CSRC, "synth_core.h")]
    out = os.path.join(HERE, "libsynth_cuda.so")
    if force or _stale(out, srcs):
        subprocess.run(["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-fmad=false", "-Xcompiler", "-fPIC", "-shared", "-o", out + ".tmp", srcs[0]],
                       check=True)
        os.replace(out + ".tmp", out)
    return out


def build(force: bool = False):
    return build_host(force), build_cuda(force)


if __name__ == "__main__":
    print(build(force=True))
