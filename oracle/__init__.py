"""CPU fp64 oracle of the DSA indexer paged MQA-logits (test infrastructure).

Only the tests, the package smoke check (``__graft_entry__.smoke``) and the
bench's CPU-baseline leg may import this module.  The product library never
loads it and shares no code with it.

The arithmetic lives in ``dsa_oracle.c`` (plain C, double precision, one loop
per index of the definition).  This module compiles it with gcc into
``oracle/_build/libdsa_oracle.so`` and wraps it with ctypes and numpy.

What it computes, for every row r (a decode request or a prefill query) and
position t < W*P::

    out[r, t] = -inf                                            if t >= L_r
              = s(t) * sum_h w[r, h] * max(0, q[r, h, :] . k(t))  otherwise

The formula's ingredients are named on "The Dispatch Wire: Connecting a
Triton Indexer Kernel to Production Inference", section "The Road to This
Message"; the cache layouts on the same page, section "The Reasoning and
Decision-Making", and on "The Dispatch Decision: Wiring a Triton Kernel into
Production", section "The Problem That Led Here"; the -inf rule on "The Final
Gate: Validating a Custom Triton Indexer Kernel Before Production
Deployment", section "What the Test Output Reveals".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdsa_oracle.so")

KV_E4M3 = 0
KV_BF16 = 1
OK = 0
BAD_ARG = 1
BAD_PAGE = 6
BAD_SEQLEN = 7

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: x86_64 and aarch64)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    lib.dsa_oracle_e4m3_to_double.restype = ctypes.c_double
    lib.dsa_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.dsa_oracle_bf16_to_double.restype = ctypes.c_double
    lib.dsa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.dsa_oracle_cpu_count.restype = ctypes.c_int
    lib.dsa_oracle_cpu_count.argtypes = []
    vp = ctypes.c_void_p
    ll = ctypes.c_longlong
    ci = ctypes.c_int
    lib.dsa_oracle_logits.restype = ci
    lib.dsa_oracle_logits.argtypes = [
        vp, vp, vp, vp, ll, ci, ci, vp, ll, vp,
        ci, ci, ci, ci, ci, vp, ll, ci]
    lib.dsa_oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.dsa_oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.dsa_oracle_kcache_store.restype = ci
    lib.dsa_oracle_kcache_store.argtypes = [vp, vp, ci, ci, ci, vp, ll, ci, ci]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB_PATH)
        return _lib


def e4m3_to_double(code: int) -> float:
    return _load().dsa_oracle_e4m3_to_double(int(code) & 0xFF)


def bf16_to_double(bits: int) -> float:
    return _load().dsa_oracle_bf16_to_double(int(bits) & 0xFFFF)


def cpu_count() -> int:
    return int(_load().dsa_oracle_cpu_count())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def logits(q_bits: np.ndarray, w: np.ndarray, kcache: np.ndarray,
           kscale_offset: int | None, page_stride: int, num_pages: int,
           kv_dtype: int, block_table: np.ndarray, bt_stride: int,
           seqlens: np.ndarray, R: int, H: int, D: int, P: int, W: int,
           nthreads: int = 0, lib=None) -> tuple[np.ndarray, int]:
    """Run the oracle.  Returns (out float64 [R, W*P], status).

    q_bits: uint16 bf16 bit patterns [R, H, D]; w: float32 [R, H];
    kcache: uint8 pool bytes (page p at byte p*page_stride);
    kscale_offset: byte offset inside the pool of page 0's fp32 scales
    (page p's at kscale_offset + p*page_stride), or None for scale 1;
    block_table: int32, row r at element r*bt_stride; seqlens: int32 [R].
    `lib` selects another compiled copy of the oracle (used by the tests
    that plant mistakes in a copy to show the pins catch them).
    """
    lib = _load() if lib is None else lib
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    kcache = np.ascontiguousarray(kcache, dtype=np.uint8)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    seqlens = np.ascontiguousarray(seqlens, dtype=np.int32)
    assert q_bits.size >= R * H * D and w.size >= R * H
    assert seqlens.size >= R
    if R > 0:
        assert block_table.size >= (R - 1) * bt_stride + W
    out = np.empty((R, W * P), dtype=np.float64)
    ks = None if kscale_offset is None else _ptr(kcache) + int(kscale_offset)
    status = lib.dsa_oracle_logits(
        _ptr(q_bits), _ptr(w), _ptr(kcache), ks, int(page_stride),
        int(num_pages), int(kv_dtype), _ptr(block_table), int(bt_stride),
        _ptr(seqlens), int(R), int(H), int(D), int(P), int(W), _ptr(out),
        int(W * P), int(nthreads))
    return out, int(status)


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code to the fp32 value x (ties to even, saturating)."""
    return int(_load().dsa_oracle_e4m3_encode(float(x)))


def kcache_store(k_bits: np.ndarray, slots: np.ndarray, kcache: np.ndarray,
                 page_stride: int, num_pages: int, kv_dtype: int, D: int = 128,
                 P: int = 64, lib=None) -> int:
    """Write the key rows k_bits (bf16 bits [n, D]) into their slots of the
    byte pool kcache (modified in place); returns the status."""
    L = lib or _load()
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    sl = np.ascontiguousarray(slots, dtype=np.int32)
    assert kcache.dtype == np.uint8 and kcache.flags.c_contiguous
    n = int(sl.shape[0])
    assert k.shape == (n, D)
    return int(L.dsa_oracle_kcache_store(_ptr(k), _ptr(sl), n, D, P, _ptr(kcache),
                                         int(page_stride), int(num_pages), int(kv_dtype)))
