"""Build step for the CPU oracle (plain C, gcc).

TEST INFRASTRUCTURE ONLY: the oracle is compiled here so that the test suite,
the smoke check and the benchmark's CPU-baseline leg can load it.  The GPU
library never links or loads it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sfar_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")

CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fno-strict-aliasing", "-Wall", "-Wextra", "-pthread"]


def build_oracle(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or one planted-mistake variant) and return the .so path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    name = "libsfar_oracle.so" if mutant == 0 else f"libsfar_oracle_mutant{mutant}.so"
    out = os.path.join(OUT_DIR, name)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DORACLE_MUTANT={int(mutant)}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(force=True))
