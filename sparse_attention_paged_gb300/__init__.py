"""GB300 (sm_103a) DSA indexer paged MQA-logits.

Thin Python binding of libdsa_indexer.so (``include/dsa_indexer.h``).  The
functions below carry the C names and only marshal arguments: tensors become
device pointers, the stream defaults to torch's current stream.  Every step
of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and a missing library raises.

For each row r and position t < W*64:
``out[r, t] = scale(t) * sum_h w[r, h] * relu(q[r, h, :] . k(t))`` if
``t < seqlens[r]``, else ``-inf``.
"""
from __future__ import annotations

import ctypes

from . import _native

KV_FP8_E4M3 = 0
KV_BF16 = 1
H = 64
D = 128
PAGE = 64

STATUS = {
    0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED",
    3: "DSA_ERR_MISALIGNED", 4: "DSA_ERR_CUDA", 5: "DSA_ERR_TIMEOUT",
    6: "DSA_ERR_BAD_PAGE", 7: "DSA_ERR_BAD_SEQLEN",
}


class DsaError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(dsa_status_string(status))


def _p(x) -> int | None:
    """Device address of a tensor, or an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor (the library takes device pointers)")
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dsa_status_string(status: int) -> str:
    return _native.load().dsa_status_string(int(status)).decode()


def dsa_indexer_abi_version() -> int:
    return int(_native.load().dsa_indexer_abi_version())


def dsa_indexer_logits_decode(q, w, kcache, kscale, page_stride_bytes, num_pages,
                              kv_dtype, block_table, bt_stride, seqlens, B, H, D,
                              page_size, W, out, out_stride, dev_status=None,
                              stream=None) -> int:
    """C ``dsa_indexer_logits_decode``; returns its status code."""
    return int(_native.load().dsa_indexer_logits_decode(
        _p(q), _p(w), _p(kcache), _p(kscale), int(page_stride_bytes), int(num_pages),
        int(kv_dtype), _p(block_table), int(bt_stride), _p(seqlens), int(B), int(H),
        int(D), int(page_size), int(W), _p(out), int(out_stride), _p(dev_status),
        _stream(stream)))


def dsa_indexer_logits_prefill(q, w, kcache, kscale, page_stride_bytes, num_pages,
                               kv_dtype, block_table, bt_stride, seqlens, n_q, H, D,
                               page_size, W, out, out_stride, dev_status=None,
                               stream=None) -> int:
    """C ``dsa_indexer_logits_prefill``; returns its status code."""
    return int(_native.load().dsa_indexer_logits_prefill(
        _p(q), _p(w), _p(kcache), _p(kscale), int(page_stride_bytes), int(num_pages),
        int(kv_dtype), _p(block_table), int(bt_stride), _p(seqlens), int(n_q), int(H),
        int(D), int(page_size), int(W), _p(out), int(out_stride), _p(dev_status),
        _stream(stream)))


def dsa_indexer_logits_prefill_varlen(q, w, kcache, kscale, page_stride_bytes, num_pages,
                                      kv_dtype, block_table, bt_stride, cu_q, seqlens, H, D,
                                      page_size, W, out, out_stride, dev_status=None,
                                      stream=None) -> int:
    """C ``dsa_indexer_logits_prefill_varlen``; returns its status code.  `cu_q`
    is host data (a sequence of n_req + 1 ints); n_req = len(cu_q) - 1."""
    offs = [int(v) for v in cu_q]
    n_req = max(len(offs) - 1, 0)
    arr = (ctypes.c_int * max(len(offs), 1))(*offs)
    return int(_native.load().dsa_indexer_logits_prefill_varlen(
        _p(q), _p(w), _p(kcache), _p(kscale), int(page_stride_bytes), int(num_pages),
        int(kv_dtype), _p(block_table), int(bt_stride),
        ctypes.cast(arr, ctypes.c_void_p).value if offs else None, n_req, _p(seqlens),
        int(H), int(D), int(page_size), int(W), _p(out), int(out_stride), _p(dev_status),
        _stream(stream)))


def dsa_indexer_topk_decode(q, w, kcache, kscale, page_stride_bytes, num_pages, kv_dtype,
                            block_table, bt_stride, seqlens, B, H, D, page_size, W, k_top,
                            topk_idx, topk_val, topk_stride, workspace, workspace_floats,
                            dev_status=None, stream=None) -> int:
    """C ``dsa_indexer_topk_decode``; returns its status code."""
    return int(_native.load().dsa_indexer_topk_decode(
        _p(q), _p(w), _p(kcache), _p(kscale), int(page_stride_bytes), int(num_pages),
        int(kv_dtype), _p(block_table), int(bt_stride), _p(seqlens), int(B), int(H), int(D),
        int(page_size), int(W), int(k_top), _p(topk_idx), _p(topk_val), int(topk_stride),
        _p(workspace), int(workspace_floats), _p(dev_status), _stream(stream)))


TOPK_AUTO = 0
TOPK_TWO_PASS = 1
TOPK_FUSED = 2


def dsa_indexer_topk_decode_form(q, w, kcache, kscale, page_stride_bytes, num_pages, kv_dtype,
                                 block_table, bt_stride, seqlens, B, H, D, page_size, W, k_top,
                                 topk_idx, topk_val, topk_stride, workspace, workspace_floats,
                                 dev_status=None, form=TOPK_AUTO, stream=None) -> int:
    """C ``dsa_indexer_topk_decode_form``; returns its status code."""
    return int(_native.load().dsa_indexer_topk_decode_form(
        _p(q), _p(w), _p(kcache), _p(kscale), int(page_stride_bytes), int(num_pages),
        int(kv_dtype), _p(block_table), int(bt_stride), _p(seqlens), int(B), int(H), int(D),
        int(page_size), int(W), int(k_top), _p(topk_idx), _p(topk_val), int(topk_stride),
        _p(workspace), int(workspace_floats), _p(dev_status), int(form), _stream(stream)))


def dsa_indexer_topk_decode_static(q, w, kcache, kscale, page_stride_bytes, num_pages,
                                   kv_dtype, block_table, bt_stride, seqlens, B, H, D,
                                   page_size, W, k_top, topk_idx, topk_val, topk_stride,
                                   dev_status=None, stream=None) -> int:
    """C ``dsa_indexer_topk_decode_static``; returns its status code."""
    return int(_native.load().dsa_indexer_topk_decode_static(
        _p(q), _p(w), _p(kcache), _p(kscale), int(page_stride_bytes), int(num_pages),
        int(kv_dtype), _p(block_table), int(bt_stride), _p(seqlens), int(B), int(H), int(D),
        int(page_size), int(W), int(k_top), _p(topk_idx), _p(topk_val), int(topk_stride),
        _p(dev_status), _stream(stream)))


def dsa_kcache_store(k, slot_mapping, n, kcache, page_stride_bytes, num_pages, kv_dtype,
                     D, page_size, dev_status=None, stream=None) -> int:
    """C ``dsa_kcache_store``; returns its status code."""
    return int(_native.load().dsa_kcache_store(
        _p(k), _p(slot_mapping), int(n), _p(kcache), int(page_stride_bytes), int(num_pages),
        int(kv_dtype), int(D), int(page_size), _p(dev_status), _stream(stream)))


def indexer_logits(kind: str, q, w, kcache, kscale, page_stride_bytes, num_pages,
                   kv_dtype, block_table, bt_stride, seqlens, W, out=None,
                   dev_status=None, stream=None):
    """Allocate the [rows, W*64] fp32 output (if not given) and run one call.

    ``kind`` is "decode" or "prefill".  Raises DsaError on a host-side error.
    """
    import torch
    rows = int(seqlens.shape[0])
    if out is None:
        out = torch.empty((rows, W * PAGE), dtype=torch.float32, device=seqlens.device)
    fn = dsa_indexer_logits_decode if kind == "decode" else dsa_indexer_logits_prefill
    st = fn(q, w, kcache, kscale, page_stride_bytes, num_pages, kv_dtype, block_table,
            bt_stride, seqlens, rows, H, D, PAGE, W, out, out.stride(0), dev_status, stream)
    if st != 0:
        raise DsaError(st)
    return out
