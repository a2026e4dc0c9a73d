"""The top-k entry point that allocates nothing, for callers that cannot
allocate device memory for a workspace (its logits go to a fixed device
array of the library).  The file name sorts last, so that a run stopping at
its first failure has run every other test first; the tests themselves do
not depend on their order (free memory is read after the call that sets the
array up).

Host part: the entry point is exported, refuses an oversized call before any
device work and validates every other argument as the workspace entry point
does.  GPU part: on two calls in a row, results bit-identical to the
workspace entry point's and a valid top-k against the oracle's logits; no
device memory taken by repeated calls; capture after the first call."""
import os
import shutil

import numpy as np
import pytest

from sparse_attention_paged_gb300 import _native
from sparse_attention_paged_gb300 import workloads as wl

needs_nvcc = pytest.mark.skipif(shutil.which(_native.NVCC) is None and
                                not os.path.exists(_native.LIB_PATH),
                                reason="nvcc not available and library not built")
A = 0x10000
MAX_FLOATS = 24 << 20


def _call(lib, **kw):
    import sparse_attention_paged_gb300 as s
    args = dict(q=A, w=A, kcache=A, kscale=A + 8192, page_stride_bytes=8448, num_pages=16,
                kv_dtype=0, block_table=A, bt_stride=8, seqlens=A, B=2, H=64, D=128,
                page_size=64, W=8, k_top=64, topk_idx=A, topk_val=A, topk_stride=64,
                dev_status=None, stream=0)
    args.update(kw)
    return s.dsa_indexer_topk_decode_static(**args)


@needs_nvcc
def test_exported():
    lib = _native.load()
    assert hasattr(lib, "dsa_indexer_topk_decode_static")
    assert "dsa_indexer_topk_decode_static" in _native.EXPORTS


@needs_nvcc
def test_oversized_call_is_refused_before_device_work():
    lib = _native.load()
    # 64 rows x 6,145 pages x 64 positions > 24 Mi floats; fake pointers:
    # nothing may be touched
    assert _call(lib, B=64, W=6145, bt_stride=6145) == 2
    assert _call(lib, B=0) == 0
    assert _call(lib, B=-1) == 1
    # with no rows nothing is launched, but the other arguments are still
    # checked as the workspace entry point checks them
    assert _call(lib, B=0, H=32) == 2
    assert _call(lib, B=0, kv_dtype=5) == 1
    assert _call(lib, B=0, k_top=0) == 1
    assert _call(lib, B=0, W=0) == 1


def _run_both(w, k):
    import torch
    import sparse_attention_paged_gb300 as lib
    from tests.parity import DeviceWorkload
    dw = DeviceWorkload(w)
    T = w.W * w.P
    outs = []
    for static in (False, True):
        idx = torch.full((w.R, k), -7, dtype=torch.int32, device="cuda")
        val = torch.full((w.R, k), 7.0, dtype=torch.float32, device="cuda")
        args = (dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w.page_stride, w.num_pages, w.kv_dtype,
                dw.bt, w.bt_stride, dw.seqlens, w.R, 64, 128, 64, w.W, k, idx, val, k)
        if static:
            st = lib.dsa_indexer_topk_decode_static(*args, dw.status)
        else:
            ws = torch.empty(w.R * T, dtype=torch.float32, device="cuda")
            st = lib.dsa_indexer_topk_decode(*args, ws, ws.numel(), dw.status)
        assert st == 0
        torch.cuda.synchronize()
        outs.append((idx.cpu().numpy(), val.cpu().numpy()))
    return dw, outs


@pytest.mark.gpu
def test_static_matches_the_workspace_call():
    from tests.test_gpu_topk import _check
    for w, k in [(wl.decode_with_lengths("na", [0, 5, 700, 2000], 40, seed=21), 64),
                 (wl.cfg3(4097), 2048)]:
        _, ((i0, v0), (i1, v1)) = _run_both(w, k)
        assert np.array_equal(i0, i1)
        assert np.array_equal(v0.view(np.uint32), v1.view(np.uint32))
        # the static call's own result is a valid top-k of the oracle's logits
        L = w.seqlens
        rows = (list(range(w.R)) if w.R <= 8 else
                sorted({int(np.argmin(L)), int(np.argmax(L)), 0, w.R - 1}))
        _check(w, k, i1, v1, rows)


@pytest.mark.gpu
def test_repeated_calls_take_no_device_memory():
    import torch
    import sparse_attention_paged_gb300 as lib
    from tests.parity import DeviceWorkload
    w = wl.decode_with_lengths("na2", [100, 3000, 64], 60, seed=22)
    dw = DeviceWorkload(w)
    k = 32
    idx = torch.empty((w.R, k), dtype=torch.int32, device="cuda")
    val = torch.empty((w.R, k), dtype=torch.float32, device="cuda")
    args = (dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w.page_stride, w.num_pages, w.kv_dtype,
            dw.bt, w.bt_stride, dw.seqlens, w.R, 64, 128, 64, w.W, k, idx, val, k, dw.status)
    assert lib.dsa_indexer_topk_decode_static(*args) == 0      # first call: the array is set up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        assert lib.dsa_indexer_topk_decode_static(*args) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(dw.status.item()) == 0


@pytest.mark.gpu
def test_static_call_captured_after_its_first_call():
    """The first call on a device (made above, outside capture) sets the
    array up; later calls may be captured and replayed with new lengths."""
    import torch
    import sparse_attention_paged_gb300 as lib
    from tests.parity import DeviceWorkload
    W, k = 50, 128
    w0 = wl.decode_with_lengths("na3", [2000, 3200, 5, 900], W, seed=23)
    w1 = wl.decode_with_lengths("na4", [3199, 64, 1700, 129], W, seed=24)
    dw = DeviceWorkload(w0)
    idx = torch.empty((w0.R, k), dtype=torch.int32, device="cuda")
    val = torch.empty((w0.R, k), dtype=torch.float32, device="cuda")
    args = lambda: (dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w0.page_stride, w0.num_pages,
                    w0.kv_dtype, dw.bt, w0.bt_stride, dw.seqlens, w0.R, 64, 128, 64, W, k, idx,
                    val, k, dw.status)
    assert lib.dsa_indexer_topk_decode_static(*args()) == 0
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lib.dsa_indexer_topk_decode_static(*args())
    for w in (w0, w1):
        src = DeviceWorkload(w)
        for name in ("q", "wt", "kcache", "bt", "seqlens"):
            getattr(dw, name).copy_(getattr(src, name))
        g.replay()
        torch.cuda.synchronize()
        got = (idx.cpu().numpy().copy(), val.cpu().numpy().copy())
        _, ((i0, v0), _) = _run_both(w, k)
        assert np.array_equal(got[0], i0)
        assert np.array_equal(got[1].view(np.uint32), v0.view(np.uint32))
