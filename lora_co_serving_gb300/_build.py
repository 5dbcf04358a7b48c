"""Build ``liblora_mixed.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Sources are compiled in parallel into ``_build/`` beside this file and linked
into ``liblora_mixed.so`` next to the package.  The CUDA runtime is linked
statically (nvcc's default), so the library needs only the driver at run time.
"""
import concurrent.futures as cf
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblora_mixed.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ["api.cu", "tc_kernel.cu", "simt.cu", "noalloc.cu", "adamw.cu"]
CXX_SOURCES = ["plan.cpp", "latency.cpp"]


def _nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _run(cmd):
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("build step failed:\n%s\n%s%s" % (" ".join(cmd), res.stdout, res.stderr))
    return res.stdout + res.stderr


def build(force=False, verbose=False, extra_flags=(), out=None, objdir=None, csrc=None):
    """Compile and link the library if any source is newer than it; return its path.

    ``extra_flags``/``out``/``objdir`` build a variant (e.g. other -D tuning values) into another file.
    """
    lib_path = out or LIB
    objdir = objdir or OBJDIR
    src_dir = csrc or CSRC
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _deps():
        return lib_path
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", src_dir, "-Xcompiler", "-fPIC"]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(objdir, src + ".o")
        jobs.append([nvcc, *ARCH, "-lineinfo", *common, *extra_flags, "-c", os.path.join(src_dir, src), "-o", obj])
    for src in CXX_SOURCES:
        obj = os.path.join(objdir, src + ".o")
        jobs.append([nvcc, *common, *extra_flags, "-x", "c++", "-c", os.path.join(src_dir, src), "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(_run, jobs))
    objs = [os.path.join(objdir, s + ".o") for s in CUDA_SOURCES + CXX_SOURCES]
    tmp = lib_path + ".tmp%d" % os.getpid()
    outs.append(_run([nvcc, *ARCH, "-shared", "-o", tmp, *objs]))
    os.replace(tmp, lib_path)
    if verbose:
        print("".join(outs))
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
