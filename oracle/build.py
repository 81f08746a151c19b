"""Build the fp64 CPU oracle (test infrastructure) into oracle/_lib/.

`build_oracle()` compiles dattn_oracle.cpp with g++ into a shared library that
the tests load with ctypes. `build_oracle(mutation=n)` builds a copy with one
known mistake planted (see the ORACLE_MUTATION blocks in the source), used only
by the tests that show each pin can fail.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dattn_oracle.cpp")
OUT_DIR = os.path.join(HERE, "_lib")


def lib_path(mutation: int = 0) -> str:
    name = "liboracle.so" if mutation == 0 else f"liboracle_mut{mutation}.so"
    return os.path.join(OUT_DIR, name)


def build_oracle(mutation: int = 0, force: bool = False) -> str:
    out = lib_path(mutation)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off",
           "-pthread", f"-DORACLE_MUTATION={mutation}", SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(int(sys.argv[1]) if len(sys.argv) > 1 else 0, force=True))
