"""Compile the C oracle into oracle/libmoe_oracle.so (test infrastructure).

The oracle is built with -O2 -ffp-contract=off and without -ffast-math so
that every binary32 operation is a single IEEE round-to-nearest-even step and
no multiply-add is contracted, on x86_64 and on aarch64 alike.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "moe_oracle.c")
LIBRARY = os.path.join(HERE, "libmoe_oracle.so")
FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall",
         "-Wextra", "-fPIC", "-shared"]


def build(force: bool = False, source: str = SOURCE, output: str = LIBRARY,
          extra_flags=()) -> str:
    """Build the oracle library if it is missing or older than its source.

    `source`, `output` and `extra_flags` exist so that tests can compile a
    deliberately altered copy of the oracle into a scratch directory."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    cc = os.environ.get("CC", "gcc")
    tmp = output + ".tmp%d" % os.getpid()
    cmd = [cc, *FLAGS, *extra_flags, "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
