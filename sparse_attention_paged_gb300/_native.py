"""Build and load libdsa_indexer.so (the sm_103a CUDA library) in-tree.

The library is compiled with nvcc for ``sm_103a`` only and loaded with
ctypes.  There is no fallback: if the library cannot be built or loaded the
calls raise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD, "libdsa_indexer.so")
NVCC = os.environ.get("NVCC", "nvcc")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]

# Every symbol include/dsa_indexer.h declares.
EXPORTS = ("dsa_indexer_logits_decode", "dsa_indexer_logits_prefill",
           "dsa_indexer_logits_prefill_varlen", "dsa_indexer_topk_decode",
           "dsa_indexer_topk_decode_form",
           "dsa_indexer_topk_decode_static", "dsa_kcache_store",
           "dsa_status_string", "dsa_indexer_abi_version")

_lib = None
_lock = threading.Lock()


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = _sources()
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu under csrc/ for sm_103a and link the shared library."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(BUILD, exist_ok=True)
    objs = []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [NVCC, *ARCH_FLAGS, *NVCC_FLAGS, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, srcs))
    for obj, log in results:
        objs.append(obj)
        if verbose and log:
            print(log)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load the library (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if is_stale():
            build()
        lib = ctypes.CDLL(LIB_PATH)
        vp, ll, ci = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int
        sig = [vp, vp, vp, vp, ll, ci, ci, vp, ll, vp, ci, ci, ci, ci, ci, vp, ll, vp, vp]
        for name in ("dsa_indexer_logits_decode", "dsa_indexer_logits_prefill"):
            fn = getattr(lib, name)
            fn.restype = ci
            fn.argtypes = sig
        lib.dsa_indexer_topk_decode.restype = ci
        lib.dsa_indexer_topk_decode.argtypes = [vp, vp, vp, vp, ll, ci, ci, vp, ll, vp, ci, ci,
                                                ci, ci, ci, ci, vp, vp, ll, vp, ll, vp, vp]
        lib.dsa_indexer_topk_decode_form.restype = ci
        lib.dsa_indexer_topk_decode_form.argtypes = [vp, vp, vp, vp, ll, ci, ci, vp, ll, vp, ci,
                                                     ci, ci, ci, ci, ci, vp, vp, ll, vp, ll, vp,
                                                     ci, vp]
        lib.dsa_indexer_logits_prefill_varlen.restype = ci
        lib.dsa_indexer_logits_prefill_varlen.argtypes = [vp, vp, vp, vp, ll, ci, ci, vp, ll, vp,
                                                          ci, vp, ci, ci, ci, ci, vp, ll, vp, vp]
        lib.dsa_indexer_topk_decode_static.restype = ci
        lib.dsa_indexer_topk_decode_static.argtypes = [vp, vp, vp, vp, ll, ci, ci, vp, ll, vp, ci,
                                                       ci, ci, ci, ci, ci, vp, vp, ll, vp, vp]
        lib.dsa_kcache_store.restype = ci
        lib.dsa_kcache_store.argtypes = [vp, vp, ci, vp, ll, ci, ci, ci, ci, vp, vp]
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_status_string.argtypes = [ci]
        lib.dsa_indexer_abi_version.restype = ci
        lib.dsa_indexer_abi_version.argtypes = []
        _lib = lib
        return lib
