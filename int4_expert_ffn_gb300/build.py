"""Compile libcoli.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each translation unit is compiled in parallel, then linked with nvcc into
``int4_expert_ffn_gb300/libcoli.so``.  A stamp of the flags and source mtimes
skips the rebuild when nothing changed.

``build(variant="check")`` makes the diagnostic bounds-checked library
``libcoli_check.so`` (``-DCOLI_CHECK``: indices derived from data are checked
against their buffers and reported through COLI_FLAG_BOUNDS) beside it; the
binding loads it instead when ``COLI_LIBRARY=check`` is set in the environment.
"""
import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcoli.so")
VARIANTS = {
    # name: (library file, build directory, extra nvcc flags)
    "": (LIB, BUILD, []),
    "check": (os.path.join(PKG, "libcoli_check.so"), os.path.join(BUILD, "check"), ["-DCOLI_CHECK"]),
}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
           "-I" + INCLUDE, "-I" + CSRC]


def _nvcc():
    nv = shutil.which("nvcc")
    if nv:
        return nv
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcoli")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stamp(srcs, extra):
    h = hashlib.sha256()
    h.update(" ".join(ARCH + NVFLAGS + extra).encode())
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(INCLUDE, "coli.h"))
    for p in sorted(deps):
        with open(p, "rb") as f:
            h.update(p.encode())
            h.update(f.read())
    return h.hexdigest()


def build(force=False, verbose=False, extra_flags=(), variant=""):
    """Build libcoli.so (or a variant of it); returns its path."""
    lib_path, build_dir, variant_flags = VARIANTS[variant]
    extra = variant_flags + list(extra_flags)
    srcs = sources()
    stamp = _stamp(srcs, extra)
    stamp_file = os.path.join(build_dir, "stamp")
    if (not force and os.path.exists(lib_path) and os.path.exists(stamp_file)
            and open(stamp_file).read() == stamp):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVFLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib_path + ".tmp.%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib_path)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                variant="check" if "--check" in sys.argv else ""))
