"""Build the C-ABI library libpa_gb300.so for sm_103a, in tree.

Each translation unit under csrc/ is compiled by nvcc in parallel and the
objects are linked into paged_kv_cache_124_gb300/libpa_gb300.so.  Nothing is
rebuilt when the library is newer than every source and header.

    python -m paged_kv_cache_124_gb300.build [--force]
"""

import concurrent.futures
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(ROOT, "_build", "obj")
LIB = os.path.join(PKG, "libpa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libpa_gb300.so")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _inputs():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sources() + hdrs + [os.path.abspath(__file__)]


# ELF e_machine of a shared object built for this host (x86-64 or AArch64)
_ELF_MACHINE = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}


def elf_matches_host(header, machine=None):
    """True if `header` (the first 20 bytes of a file) starts a 64-bit
    little-endian ELF object for this host's machine."""
    want = _ELF_MACHINE.get((machine or platform.machine()).lower())
    return (len(header) >= 20 and header[:4] == b"\x7fELF" and header[4] == 2 and header[5] == 1 and
            want is not None and int.from_bytes(header[18:20], "little") == want)


def up_to_date():
    """The library exists, was built for this host's machine, and is newer
    than every source and header."""
    if not os.path.exists(LIB):
        return False
    with open(LIB, "rb") as f:
        if not elf_matches_host(f.read(20)):
            return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _compile(src, verbose):
    obj = os.path.join(OBJ_DIR, os.path.basename(src) + ".o")
    cmd = [_nvcc(), *ARCH, *COMMON, "-c", src, "-o", obj]
    if src.endswith(".cu") and verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj, r.stderr


def build(force=False, verbose=False):
    """Compile csrc/ into libpa_gb300.so (sm_103a).  Returns the library path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), sources()))
    if verbose:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
