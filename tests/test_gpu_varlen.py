"""GPU parity of the varlen prefill (a block-table row per request; the
query-tile kernel over up to 128 requests per launch) through the C ABI,
against the oracle.  The
oracle reads the workload's per-query rows (copies of each request's row);
the call gets one row per request and the request offsets."""
import numpy as np
import pytest

from sparse_attention_paged_gb300 import workloads as wl
from tests.parity import DeviceWorkload, compare, oracle_rows

pytestmark = pytest.mark.gpu


def _run_varlen(w, shared_row=False):
    import torch
    import sparse_attention_paged_gb300 as lib
    dw = DeviceWorkload(w)
    cu, req_bt = wl.request_tables(w)
    if shared_row:
        req_bt = req_bt[:1]
    bt = torch.from_numpy(np.ascontiguousarray(req_bt)).cuda()
    st = lib.dsa_indexer_logits_prefill_varlen(
        dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w.page_stride, w.num_pages, w.kv_dtype, bt,
        0 if shared_row else w.W, cu, dw.seqlens, 64, 128, 64, w.W, dw.out, dw.out.stride(0),
        dw.status)
    assert st == 0
    torch.cuda.synchronize()
    return dw


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_E4M3])
def test_varlen_small_full(kv):
    # an empty request, a one-token request, ragged query tiles, a request
    # of several query tiles
    w = wl.prefill_varlen("vl_small", [(5, 300), (0, 64), (70, 1000), (1, 65), (9, 200)],
                          seed=41, kv_dtype=kv)
    dw = _run_varlen(w)
    assert int(dw.status.item()) == 0
    ref, st = oracle_rows(w)
    assert st == 0
    compare(dw.out.cpu().numpy(), ref)


def test_varlen_fp8_two_requests_full():
    w = wl.prefill_varlen("vl_fp8", [(64, 2048), (200, 5000)], seed=42, kv_dtype=wl.KV_E4M3)
    dw = _run_varlen(w)
    assert int(dw.status.item()) == 0
    ref, st = oracle_rows(w)
    assert st == 0
    compare(dw.out.cpu().numpy(), ref)


def test_varlen_one_row_shared_by_every_request():
    # bt_stride = 0: every request reads table row 0; the oracle is given
    # the same row for every query
    w = wl.prefill_varlen("vl_shared", [(12, 640), (30, 640), (3, 640)], seed=43)
    w.block_table[:] = w.block_table[0]
    dw = _run_varlen(w, shared_row=True)
    assert int(dw.status.item()) == 0
    ref, st = oracle_rows(w)
    assert st == 0
    compare(dw.out.cpu().numpy(), ref)


def test_config6_through_request_rows_sampled():
    w = wl.cfg6()
    dw = _run_varlen(w)
    assert int(dw.status.item()) == 0
    o = dw.out.cpu().numpy()
    T = w.W * w.P
    L = np.clip(w.seqlens.astype(np.int64), 0, T)
    assert np.array_equal(np.isneginf(o), np.arange(T)[None, :] >= L[:, None])
    assert not np.isnan(o).any()
    rows = []
    for a, n in w.meta["groups"]:            # first, middle and last token of every request
        rows += [a, a + n // 2, a + n - 1]
    rows = sorted(rows)
    ref, st = oracle_rows(w, rows)
    assert st == 0
    compare(o[rows], ref)


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_E4M3])
def test_varlen_more_requests_than_one_launch_takes(kv):
    """131 requests: two launches (128 requests, then 3), with empty and
    one-token requests on both sides of the boundary."""
    g = np.random.default_rng(7)
    reqs = []
    for b in range(131):
        n = int(g.integers(0, 7))
        if b in (0, 127, 128, 130):
            n = 0 if b in (0, 128) else 1
        c = int(g.integers(max(n, 1), 260))
        reqs.append((n, c))
    w = wl.prefill_varlen("vl_many", reqs, seed=44, kv_dtype=kv)
    dw = _run_varlen(w)
    assert int(dw.status.item()) == 0
    ref, st = oracle_rows(w)
    assert st == 0
    compare(dw.out.cpu().numpy(), ref)
