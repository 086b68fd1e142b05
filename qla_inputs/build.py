"""Builds the input generator library (plain C, gcc) in-tree."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def library_path():
    return os.path.join(HERE, "_lib", "libqla_inputs.so")


def build_command():
    src = os.path.join(HERE, "gen.c")
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
            src, "-o", library_path(), "-lm"]


def build():
    os.makedirs(os.path.dirname(library_path()), exist_ok=True)
    subprocess.run(build_command(), check=True)
    return library_path()
