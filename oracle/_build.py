"""Build liboracle.so in place with gcc (plain C, fp64, no FMA contraction).

TEST INFRASTRUCTURE: the oracle is only loaded by the tests, the smoke check and
the bench's CPU-baseline leg.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = [os.path.join(HERE, "oracle.c")]
DEPS = SRC + [os.path.join(HERE, "oracle.h")]
OUT = os.path.join(HERE, "liboracle.so")


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build_oracle(force: bool = False) -> str:
    if not force and not _stale(OUT, DEPS):
        return OUT
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", OUT + ".tmp"] + SRC + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(OUT + ".tmp", OUT)
    return OUT


if __name__ == "__main__":
    print(build_oracle(force=True))
