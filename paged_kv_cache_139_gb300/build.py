"""Build libpkv.so in-tree: CUDA sources for sm_103a with nvcc, the host
allocator with g++, linked into paged_kv_cache_139_gb300/lib/libpkv.so."""
from __future__ import annotations

import os
import pathlib
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OBJ = PKG / "_build"
LIBDIR = PKG / "lib"
LIB = LIBDIR / "libpkv.so"

CUDA_SOURCES = ["runtime.cu", "cache_ops.cu", "attention.cu", "attention_noalloc.cu", "prefill.cu"]
CXX_SOURCES = ["allocator.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> pathlib.Path:
    nvcc = shutil.which("nvcc")
    if nvcc:
        return pathlib.Path(nvcc).resolve().parent.parent
    return pathlib.Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))


def _nvcc() -> str:
    return str(_cuda_home() / "bin" / "nvcc")


def _sources(src_dir: pathlib.Path = CSRC):
    return [src_dir / s for s in CUDA_SOURCES + CXX_SOURCES]


def _headers():
    return list(CSRC.glob("*.h")) + list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > t for p in _sources() + _headers() + [pathlib.Path(__file__)])


def _compile(src: pathlib.Path, verbose: bool, obj_dir: pathlib.Path = OBJ, defines=()) -> pathlib.Path:
    obj = obj_dir / (src.name + ".o")
    if src.suffix == ".cu":
        cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", str(INCLUDE), "-I", str(src.parent), *[f"-D{d}" for d in defines], "-c", str(src), "-o",
               str(obj)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
    else:
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", str(INCLUDE), "-I", str(src.parent),
               "-I", str(_cuda_home() / "include"), "-c", str(src), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, out: pathlib.Path = None, defines=(),
          src_dir: pathlib.Path = CSRC) -> pathlib.Path:
    """Build the library (by default in-tree); `out`, `defines` and `src_dir`
    build a variant (tuning knobs set, or another source tree) elsewhere."""
    lib = LIB if out is None else pathlib.Path(out)
    if out is None and not defines and not force and not _stale():
        return LIB
    obj_dir = OBJ if out is None else lib.parent / "_obj"
    obj_dir.mkdir(parents=True, exist_ok=True)
    lib.parent.mkdir(parents=True, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(_sources())) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, obj_dir, defines), _sources(pathlib.Path(src_dir))))
    tmp = lib.parent / f"libpkv.{os.getpid()}.so"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs), "-lcudart_static", "-lrt", "-ldl",
           "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
