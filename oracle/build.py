"""Build step for the fp64 CPU oracle (test infrastructure only).

Compiles ``gdn_oracle.c`` with gcc into ``oracle/_build/liboracle.so``.  The
oracle is plain C11 + POSIX threads, so the same command builds it on x86-64
and on aarch64 hosts.  ``mutant=k`` builds the k-th planted-mistake variant,
used only by the tests that show the pins catch such mistakes.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")


def lib_path(mutant=0):
    name = "liboracle.so" if not mutant else f"liboracle_mutant{mutant}.so"
    return os.path.join(BUILD_DIR, name)


def build_oracle(mutant=0, force=False):
    """Compile the oracle (or one mutant) if it is missing or stale; return its path."""
    out = lib_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC)):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread",
           f"-DORACLE_MUTANT={int(mutant)}", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(force=True))
