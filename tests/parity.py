"""Helpers shared by the parity tests: move a workload to the GPU, run the
library through the C ABI, run the oracle on the same bytes, compare."""
from __future__ import annotations

import numpy as np

import oracle
from sparse_attention_paged_gb300 import workloads as wl

# The bar: the -inf mask agrees exactly; finite logits agree to
# max|d| <= 1e-3 * max|logit| over the call's finite entries.
REL_TOL = 1e-3


class DeviceWorkload:
    """Device copies of a Workload's inputs plus a preallocated output."""

    def __init__(self, w: wl.Workload, device="cuda"):
        import torch
        self.w = w
        self.q = torch.from_numpy(w.q_bits.view(np.int16)).to(device)
        self.wt = torch.from_numpy(w.w).to(device)
        self.kcache = torch.from_numpy(w.kcache).to(device)
        self.bt = torch.from_numpy(w.block_table).to(device)
        self.seqlens = torch.from_numpy(w.seqlens).to(device)
        self.out = torch.empty((w.R, w.W * w.P), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    @property
    def kscale_ptr(self):
        if self.w.kscale_offset is None:
            return None
        return self.kcache.data_ptr() + self.w.kscale_offset

    def call(self, stream=None, out=None, seqlens=None, bt=None) -> int:
        import sparse_attention_paged_gb300 as lib
        w = self.w
        out = self.out if out is None else out
        fn = (lib.dsa_indexer_logits_decode if w.kind == "decode"
              else lib.dsa_indexer_logits_prefill)
        return fn(self.q, self.wt, self.kcache, self.kscale_ptr, w.page_stride,
                  w.num_pages, w.kv_dtype, self.bt if bt is None else bt, w.bt_stride,
                  self.seqlens if seqlens is None else seqlens, w.R, w.H, w.D, w.P,
                  w.W, out, out.stride(0), self.status, stream)


def oracle_rows(w: wl.Workload, rows=None, nthreads=0):
    """Oracle output for all rows, or for the listed rows only."""
    if rows is None:
        rows = np.arange(w.R)
    rows = np.asarray(rows)
    q = w.q_bits[rows]
    ww = w.w[rows]
    seq = w.seqlens[rows]
    bt = w.block_table if w.bt_stride == 0 else w.block_table[rows]
    out, st = oracle.logits(q, ww, w.kcache, w.kscale_offset, w.page_stride,
                            w.num_pages, w.kv_dtype, bt, w.bt_stride, seq,
                            len(rows), w.H, w.D, w.P, w.W, nthreads=nthreads)
    return out, st


def compare(gpu: np.ndarray, ref: np.ndarray, tol: float = REL_TOL) -> dict:
    """Assert the parity bar; return the error figures."""
    gpu = np.asarray(gpu, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.array_equal(np.isneginf(gpu), np.isneginf(ref)), "-inf mask differs"
    assert np.array_equal(np.isnan(gpu), np.isnan(ref)), "NaN set differs"
    assert not np.isposinf(gpu).any()
    fin = np.isfinite(ref)
    if not fin.any():
        return {"max_abs": 0.0, "max_ref": 0.0, "rel": 0.0}
    d = np.abs(gpu[fin] - ref[fin])
    mref = float(np.abs(ref[fin]).max())
    mad = float(d.max())
    assert mad <= tol * mref, f"max|d| {mad:.3e} > {tol} * max|logit| {mref:.3e}"
    return {"max_abs": mad, "max_ref": mref, "rel": mad / mref if mref else 0.0}
