"""Build the CUDA library in-tree with nvcc (sm_103a only, no cmake)."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libexact_attn.so")
SOURCES = ["api_common.cu", "attn_api.cu", "attn_bwd_api.cu", "attn_fp8_api.cu", "rowwise_api.cu", "plan.cpp",
           "split_policy.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "exact_attn.h")]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, defines: dict | None = None, lib_path: str = LIB_PATH) -> str:
    """Compile every source to an object in parallel, then link the shared library.

    `defines` adds -D flags (compile-time variants of the kernels, e.g.
    ELS_EXP2_POLY_PER32); such a variant is linked to `lib_path`, beside the
    default library."""
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _deps_mtime():
        return lib_path
    cc = nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")] + ARCH
    common += [f"-D{k}={v}" for k, v in sorted((defines or {}).items())]
    objs = []
    tag = os.path.basename(lib_path)

    def compile_one(src):
        obj = os.path.join(LIB_DIR, src + f".{tag}.{os.getpid()}.o")
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + common
        if src.endswith(".cu") and verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-shared", "-o", tmp] + objs + ARCH + ["-lcudart"], capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_variant(name: str, defines: dict, force: bool = False) -> str:
    """A compile-time variant of the library, linked to _lib/libexact_attn_<name>.so."""
    return build(force=force, defines=defines, lib_path=os.path.join(LIB_DIR, f"libexact_attn_{name}.so"))


if __name__ == "__main__":
    print(build(force=True, verbose=True))
