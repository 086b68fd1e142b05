"""Builds the CUDA library libqla.so in-tree for sm_103a (nvcc, no cmake).

Each translation unit compiles in its own nvcc process, in parallel, then one
link step makes the shared library.  The library links the CUDA runtime
statically and resolves driver entry points at run time, so it loads on a
machine without a GPU (the exports can be checked there) and runs on GB300.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_lib", "obj")
GENCODE = "arch=compute_103a,code=sm_103a"


def library_path():
    return os.path.join(HERE, "_lib", "libqla.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def compile_flags(extra=()):
    return ["-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
            *extra]


def _compile(src, extra, objdir=OBJ):
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *compile_flags(extra), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
    return obj, r.stderr


def build(extra=(), verbose=False, out=None):
    """Compiles and links the library; `extra` adds nvcc flags, `out` writes a
    variant build to another path (its objects go to a sibling folder)."""
    objdir = OBJ if out is None else out + ".obj"
    os.makedirs(objdir, exist_ok=True)
    srcs = sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, objdir), srcs))
    if verbose:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    objs = [o for o, _ in results]
    out = out or library_path()
    tmp = out + ".tmp"
    cmd = [nvcc(), "-gencode", GENCODE, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static",
           *objs, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(extra=sys.argv[1:], verbose=True))
