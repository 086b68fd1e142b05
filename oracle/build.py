"""Builds the fp64 oracle (plain C, gcc) in-tree.  Test infrastructure only."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def library_path(variant: str = ""):
    return os.path.join(HERE, "_lib", f"libqla_oracle{variant}.so")


SOURCES = ("qla_oracle.c", "qla_local_oracle.c")


def build_command(defines=(), variant: str = ""):
    srcs = [os.path.join(HERE, s) for s in SOURCES]
    return (["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]
            + [f"-D{d}" for d in defines] + srcs + ["-o", library_path(variant), "-lm"])


def build(defines=(), variant: str = ""):
    os.makedirs(os.path.join(HERE, "_lib"), exist_ok=True)
    subprocess.run(build_command(defines, variant), check=True)
    return library_path(variant)
