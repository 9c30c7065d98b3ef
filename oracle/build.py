"""Compile the C++ oracle (nvfp4_oracle.cpp) into liboracle.so next to this
file: g++ -std=c++17 -O3 -fopenmp -ffp-contract=off, no fast-math, so that
every fp32 step of the quantiser is the single IEEE operation it names.
Test infrastructure only (see __init__.py)."""
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4_oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")
FLAGS = ["-std=c++17", "-O3", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
         "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    cxx = os.environ.get("CXX") or shutil.which("g++") or "g++"
    h = hashlib.sha256(open(SRC, "rb").read() + repr(FLAGS).encode()).hexdigest()
    stamp = LIB + ".stamp"
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == h:
        return LIB
    tmp = LIB + ".tmp"
    r = subprocess.run([cxx, *FLAGS, SRC, "-o", tmp], stdout=subprocess.PIPE,
                       stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(h)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
