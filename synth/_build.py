"""Build libfwsynth.so in place with nvcc (host loops + sm_103a fill kernels)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = [os.path.join(HERE, "synth.cu")]
DEPS = SRC + [os.path.join(HERE, "synth_rng.h")]
OUT = os.path.join(HERE, "libfwsynth.so")


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build_synth(force: bool = False) -> str:
    if not force and not _stale(OUT, DEPS):
        return OUT
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
           "-shared", "-Xcompiler", "-fPIC,-fopenmp", "-lgomp", "-o", OUT + ".tmp"] + SRC
    subprocess.run(cmd, check=True)
    os.replace(OUT + ".tmp", OUT)
    return OUT


if __name__ == "__main__":
    print(build_synth(force=True))
