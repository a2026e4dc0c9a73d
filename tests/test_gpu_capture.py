"""Every call captured in a CUDA graph and replayed after its inputs change
in place (lengths, tables, queries, keys, rows to store): the replays must
give what the oracle gives for the new inputs.  The calls' grids depend on
their shapes only, so one capture serves any lengths and tables; the
varlen prefill's request offsets are host data fixed at capture."""
import numpy as np
import pytest

import oracle
from sparse_attention_paged_gb300 import workloads as wl
from tests.parity import DeviceWorkload, compare, oracle_rows
from tests.test_gpu_topk import _check as check_topk

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Run fn once on a side stream (set-up outside capture), then capture it."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _load(dw, w):
    """w's inputs into dw's device buffers (same shapes)."""
    import torch
    src = DeviceWorkload(w)
    for name in ("q", "wt", "kcache", "bt", "seqlens"):
        dst, new = getattr(dw, name), getattr(src, name)
        assert dst.shape == new.shape
        dst.copy_(new)
    torch.cuda.synchronize()


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_E4M3])
def test_prefill_shared_table_replayed_with_new_lengths(kv):
    import torch
    w0 = wl.prefill_causal("cap_pf0", 37, 9, 200, seed=51, kv_dtype=kv)
    w1 = wl.prefill_causal("cap_pf1", 37, 9, 470, seed=52, kv_dtype=kv)
    dw = DeviceWorkload(w0)
    g = _capture(lambda: dw.call())
    g.replay()
    torch.cuda.synchronize()
    compare(dw.out.cpu().numpy(), oracle_rows(w0)[0])
    _load(dw, w1)
    g.replay()
    torch.cuda.synchronize()
    compare(dw.out.cpu().numpy(), oracle_rows(w1)[0])
    assert int(dw.status.item()) == 0


def test_varlen_prefill_replayed_with_new_lengths():
    import torch
    import sparse_attention_paged_gb300 as lib
    w = wl.prefill_varlen("cap_vl", [(9, 500), (0, 64), (30, 900)], seed=53)
    dw = DeviceWorkload(w)
    cu, req = wl.request_tables(w)
    bt = torch.from_numpy(np.ascontiguousarray(req)).cuda()

    def call():
        assert lib.dsa_indexer_logits_prefill_varlen(
            dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w.page_stride, w.num_pages, w.kv_dtype, bt,
            w.W, cu, dw.seqlens, 64, 128, 64, w.W, dw.out, dw.out.stride(0), dw.status) == 0

    g = _capture(call)
    g.replay()
    torch.cuda.synchronize()
    compare(dw.out.cpu().numpy(), oracle_rows(w)[0])
    # shorter causal limits, new queries: same buffers, same graph
    w.seqlens = np.maximum(w.seqlens - np.arange(w.R, dtype=w.seqlens.dtype) % 97, 0)
    w.q_bits = wl.prefill_varlen("cap_vl2", [(9, 500), (0, 64), (30, 900)], seed=54).q_bits
    dw.seqlens.copy_(torch.from_numpy(w.seqlens))
    dw.q.copy_(torch.from_numpy(w.q_bits.view(np.int16)))
    g.replay()
    torch.cuda.synchronize()
    compare(dw.out.cpu().numpy(), oracle_rows(w)[0])
    assert int(dw.status.item()) == 0


def test_topk_replayed_with_new_lengths():
    import torch
    import sparse_attention_paged_gb300 as lib
    W, k = 60, 300
    w0 = wl.decode_with_lengths("cap_tk0", [3000, 10, 3839, 301, 1500], W, seed=55)
    w1 = wl.decode_with_lengths("cap_tk1", [77, 3840, 2000, 300, 2999], W, seed=56)
    dw = DeviceWorkload(w0)
    idx = torch.empty((w0.R, k), dtype=torch.int32, device="cuda")
    val = torch.empty((w0.R, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(w0.R * W * 64, dtype=torch.float32, device="cuda")

    def call():
        assert lib.dsa_indexer_topk_decode(
            dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w0.page_stride, w0.num_pages, w0.kv_dtype,
            dw.bt, w0.bt_stride, dw.seqlens, w0.R, 64, 128, 64, W, k, idx, val, k, ws,
            ws.numel(), dw.status) == 0

    g = _capture(call)
    for w in (w0, w1):
        _load(dw, w)
        g.replay()
        torch.cuda.synchronize()
        check_topk(w, k, idx.cpu().numpy(), val.cpu().numpy(), list(range(w.R)))
    assert int(dw.status.item()) == 0


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_store_replayed_with_new_rows(kv):
    import torch
    import sparse_attention_paged_gb300 as lib
    s0 = wl.store_rows("cap_st0", 500, 20, seed=57, kv_dtype=kv, n_skip=7)
    s1 = wl.store_rows("cap_st1", 500, 20, seed=58, kv_dtype=kv, n_skip=3)
    k = torch.from_numpy(s0.k_bits.view(np.int16)).cuda()
    sl = torch.from_numpy(s0.slots).cuda()
    kc = torch.from_numpy(s0.kcache.copy()).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        assert lib.dsa_kcache_store(k, sl, s0.n, kc, s0.page_stride, s0.num_pages, s0.kv_dtype,
                                    128, 64, status) == 0

    g = _capture(call)
    pool = s0.kcache.copy()
    for s in (s0, s1):
        k.copy_(torch.from_numpy(s.k_bits.view(np.int16)))
        sl.copy_(torch.from_numpy(s.slots))
        g.replay()
        torch.cuda.synchronize()
        assert oracle.kcache_store(s.k_bits, s.slots, pool, s.page_stride, s.num_pages,
                                   s.kv_dtype) == 0
        assert np.array_equal(kc.cpu().numpy(), pool)
    assert int(status.item()) == 0
