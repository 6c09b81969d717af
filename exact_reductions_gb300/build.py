"""Build libvmx (CUDA, sm_103a) and its CPU test model in-tree.

nvcc compiles each translation unit for sm_103a only; the objects are linked
into ``exact_reductions_gb300/_build/libvmx.so`` against the shared CUDA
runtime. The CPU model of the ordered-sum steps (tests only) is compiled with
g++ into ``_build/libvmx_model.so``. Translation units build in parallel.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CU_SOURCES = ["vmx_kernels.cu", "vmx_intpsnr.cu"]
CPP_SOURCES = ["vmx_abi.cpp"]
HEADERS = ["ordsum.cuh", "vmx_internal.h", "vmx_intpsnr.h"]

LIB = os.path.join(BUILD, "libvmx.so")
MODEL = os.path.join(BUILD, "libvmx_model.so")


def _newer(out: str, deps: List[str]) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(d) <= t for d in deps if os.path.exists(d))


def _run(cmd: List[str]) -> None:
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        sys.stderr.write(proc.stdout + proc.stderr)
        raise RuntimeError("build step failed: " + " ".join(cmd))


def _deps() -> List[str]:
    files = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "vmx.h"))
    files.append(os.path.abspath(__file__))
    return files


def nvcc_flags(extra: List[str] = ()) -> List[str]:
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-Wall", f"-I{INCLUDE}", f"-I{CSRC}", "--expt-relaxed-constexpr",
            "-Xptxas", "-warn-spills", *extra]


def build_lib(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libvmx.so; return its path."""
    if not shutil.which(NVCC) and not os.path.exists(NVCC):
        raise RuntimeError(f"nvcc not found at {NVCC}")
    os.makedirs(BUILD, exist_ok=True)
    if not force and _newer(LIB, _deps()):
        return LIB
    objs = []
    cmds = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        cmds.append([NVCC, *nvcc_flags(), "-c", os.path.join(CSRC, src), "-o", obj])
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        cmds.append([NVCC, *nvcc_flags(), "-x", "cu", "-c", os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        list(ex.map(_run, cmds))
    tmp = LIB + f".tmp{os.getpid()}"
    _run([NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
          "-Xlinker", f"-rpath,{CUDA_HOME}/lib64"])
    os.replace(tmp, LIB)
    if verbose:
        print("built", LIB)
    return LIB


def build_variant(name: str, defines: List[str], force: bool = False) -> str:
    """Compile libvmx with extra ``-D`` defines (compile-time alternatives of
    the kernel, e.g. ``VMX_STAGES=3``) into ``_build/variants/<name>/``;
    return the library's path."""
    out = os.path.join(BUILD, "variants", name)
    os.makedirs(out, exist_ok=True)
    lib = os.path.join(out, "libvmx.so")
    if not force and _newer(lib, _deps()):
        return lib
    flags = nvcc_flags([f"-D{d}" for d in defines])
    objs, cmds = [], []
    for src, lang in [(s, []) for s in CU_SOURCES] + [(s, ["-x", "cu"]) for s in CPP_SOURCES]:
        obj = os.path.join(out, src + ".o")
        objs.append(obj)
        cmds.append([NVCC, *flags, *lang, "-c", os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        list(ex.map(_run, cmds))
    tmp = lib + f".tmp{os.getpid()}"
    _run([NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
          "-Xlinker", f"-rpath,{CUDA_HOME}/lib64"])
    os.replace(tmp, lib)
    return lib


def build_model(force: bool = False) -> str:
    """Compile the CPU model of the ordered-sum steps (tests only)."""
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(CSRC, "model", "vmx_model.cpp")
    deps = [src, os.path.join(CSRC, "ordsum.cuh"), os.path.abspath(__file__)]
    if not force and _newer(MODEL, deps):
        return MODEL
    tmp = MODEL + f".tmp{os.getpid()}"
    _run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
          "-DVMX_MODEL_MUTATIONS", "-Wall", "-Wextra", src, "-o", tmp])
    os.replace(tmp, MODEL)
    return MODEL


def ptxas_report() -> str:
    """Registers, spills and shared memory per kernel (``-Xptxas -v``)."""
    out = []
    for src in CU_SOURCES:
        proc = subprocess.run([NVCC, *nvcc_flags(["-Xptxas", "-v"]), "-c",
                               os.path.join(CSRC, src), "-o", os.devnull],
                              capture_output=True, text=True)
        out.append(proc.stderr)
    return "\n".join(out)


if __name__ == "__main__":
    if "--ptxas" in sys.argv:
        print(ptxas_report())
    else:
        print(build_lib(force="--force" in sys.argv, verbose=True))
        print(build_model(force="--force" in sys.argv))
