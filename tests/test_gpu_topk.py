"""GPU parity of decode with top-k selection, through the C ABI, against the
oracle's fp64 logits.  Positions whose logits sit within the parity
tolerance of the k-th largest may be ordered either way, so the check is
that the selection is a valid top-k: every selected position's oracle logit
is at least the k-th largest minus the tolerance, every unselected valid
position's at most it plus the tolerance; the returned values match the
oracle's; positions are distinct, increasing and valid."""
import numpy as np
import pytest

from sparse_attention_paged_gb300 import workloads as wl
from tests.parity import REL_TOL, DeviceWorkload, oracle_rows

pytestmark = pytest.mark.gpu


def _topk(w, k, rows=None):
    import torch
    import sparse_attention_paged_gb300 as lib
    dw = DeviceWorkload(w)
    T = w.W * w.P
    idx = torch.full((w.R, k), -7, dtype=torch.int32, device="cuda")
    val = torch.full((w.R, k), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(w.R * T, dtype=torch.float32, device="cuda")
    st = lib.dsa_indexer_topk_decode(dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w.page_stride,
                                     w.num_pages, w.kv_dtype, dw.bt, w.bt_stride, dw.seqlens,
                                     w.R, 64, 128, 64, w.W, k, idx, val, k, ws, ws.numel(),
                                     dw.status)
    assert st == 0
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), int(dw.status.item())


def _check(w, k, idx, val, rows):
    ref, _ = oracle_rows(w, rows)
    T = w.W * w.P
    for j, r in enumerate(rows):
        L = int(w.seqlens[r])
        ir, vr = idx[r], val[r]
        if L > T:                                    # an over-long row selects nothing
            assert (ir == -1).all() and np.isneginf(vr).all()
            continue
        L = max(L, 0)
        n = min(k, L)
        assert (ir[n:] == -1).all() and np.isneginf(vr[n:]).all()
        sel = ir[:n]
        assert (np.diff(sel) > 0).all() and (sel >= 0).all() and (sel < L).all()
        v = ref[j, :L]
        if L == 0:
            continue
        tol = REL_TOL * float(np.abs(v).max())
        assert np.abs(vr[:n] - v[sel]).max() <= tol
        if L <= k:
            assert np.array_equal(sel, np.arange(L))
            continue
        thr = np.sort(v)[::-1][k - 1]
        mask = np.ones(L, bool)
        mask[sel] = False
        assert v[sel].min() >= thr - tol, (r, v[sel].min(), thr)
        assert v[mask].max() <= thr + tol, (r, v[mask].max(), thr)


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
@pytest.mark.parametrize("k", [1, 64, 300])
@pytest.mark.parametrize("W", [40, 90])             # per-request and balanced decode modes
def test_topk_small(kv, k, W):
    T = W * 64
    lens = [0, 1, 63, k, k + 1, 700, T - 1, T, 2 * k]
    w = wl.decode_with_lengths(f"tk{k}", lens, W, seed=12 + k, kv_dtype=kv)
    idx, val, st = _topk(w, k)
    assert st == 0
    _check(w, k, idx, val, list(range(w.R)))


def test_topk_over_long_row():
    w = wl.decode_with_lengths("tk_bad", [100, 3 * 64 + 5, 5000 % 192], 3, seed=13)
    idx, val, st = _topk(w, 16)
    assert st == 7
    _check(w, 16, idx, val, [0, 1, 2])


def test_topk_config3_sampled_rows():
    w = wl.cfg3(4097)
    idx, val, st = _topk(w, 2048)
    assert st == 0
    L = w.seqlens
    rows = sorted(set([int(np.argmin(L)), int(np.argmax(L)), 0, 1, 17, 63]))
    _check(w, 2048, idx, val, rows)


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_topk_ties_take_the_lowest_positions(kv):
    """Rows whose k-th largest logit is shared by many positions: an
    all-zero query (every logit 0, so the first k positions); zeroed key
    pages under the first 3,008 positions of a row (more copies of the k-th
    value than the kernel collects); and zeroed pages under the first 512
    positions of a row with k set so that the k-th largest is one of them
    (collected, but too many to rank directly)."""
    W, k = 120, 2048
    lens = [5000, 5000, 3000, 2049, 7500]
    w = wl.decode_with_lengths("tk_ties", lens, W, seed=31, kv_dtype=kv)
    w.q_bits[0] = 0
    w.q_bits[3] = 0
    zero_pages = {1: 47, 4: 8}
    for r, n in zero_pages.items():
        for pg in w.block_table[r, :n]:
            base = int(pg) * w.page_stride
            w.kcache[base: base + (8192 if kv == wl.KV_E4M3 else 16384)] = 0
    ref, _ = oracle_rows(w, [1, 4])

    def zeros_taken_first(r, v, sel, k):
        n_pos = int((v > 0).sum())
        assert (v[:64 * zero_pages[r]] == 0).all()
        assert n_pos < k <= n_pos + 64 * zero_pages[r]   # the k-th largest is a zero
        # the zeros taken are the lowest-numbered ones (positions 0, 1, ...);
        # a logit within rounding of 0 may trade places with a zero
        taken = sel[v[sel] == 0]
        assert np.array_equal(taken, np.arange(len(taken)))
        assert abs(len(taken) - (k - n_pos)) <= 2

    idx, val, st = _topk(w, k)
    assert st == 0
    _check(w, k, idx, val, list(range(w.R)))
    for r in (0, 3):
        assert np.array_equal(idx[r], np.arange(k))
        assert (val[r] == 0).all()
    zeros_taken_first(1, ref[0, :lens[1]], idx[1], k)

    v4 = ref[1, :lens[4]]
    k4 = int((v4 > 0).sum()) + 256
    idx, val, st = _topk(w, k4)
    assert st == 0
    _check(w, k4, idx, val, [4])
    zeros_taken_first(4, v4, idx[4], k4)


def test_topk_rows_longer_than_the_shared_cache():
    """Rows past the shared-memory row cache (about 51K logits) are read
    from global memory in every pass; past 65,536 the in-order write
    evaluates every key."""
    W = 1100
    lens = [60000, 52100, 3000, 64000, 70000]
    w = wl.decode_with_lengths("tk_long", lens, W, seed=32)
    for k in (64, 2048):
        idx, val, st = _topk(w, k)
        assert st == 0
        _check(w, k, idx, val, list(range(w.R)))


@pytest.mark.parametrize("k", [64, 300])
def test_topk_more_rows_than_pairs_of_sms(k):
    """More than half as many rows as SMs: one CTA per row instead of a
    cluster of two."""
    W = 20
    g = np.random.default_rng(5)
    lens = [int(x) for x in g.integers(0, W * 64 + 1, 100)]
    lens[:4] = [0, k, k + 1, W * 64]
    w = wl.decode_with_lengths(f"tk_many{k}", lens, W, seed=33)
    idx, val, st = _topk(w, k)
    assert st == 0
    _check(w, k, idx, val, list(range(w.R)))


# --- the fused form (selection in the decode epilogue, then a merge) against
# the two-pass form: the same positions and bit-identical logits ---------------

def _fused_ws_floats(B, W, k):
    import torch
    ctas = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    hdr = (B + 1 + 3) // 4 * 4
    return hdr + (ctas + B + (B * W + 31) // 32) * (4 + 2 * k)


def _topk_form(w, k, form, ws_floats=None):
    import torch
    import sparse_attention_paged_gb300 as lib
    dw = DeviceWorkload(w)
    T = w.W * w.P
    n = max(w.R * T, ws_floats or 0)
    idx = torch.full((w.R, k), -7, dtype=torch.int32, device="cuda")
    val = torch.full((w.R, k), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.full((n,), 3.0, dtype=torch.float32, device="cuda")
    st = lib.dsa_indexer_topk_decode_form(dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w.page_stride,
                                          w.num_pages, w.kv_dtype, dw.bt, w.bt_stride, dw.seqlens,
                                          w.R, 64, 128, 64, w.W, k, idx, val, k, ws, n,
                                          dw.status, form)
    torch.cuda.synchronize()
    return st, idx.cpu().numpy(), val.cpu().numpy(), int(dw.status.item())


def _same_as_two_pass(w, k, expect_status=0):
    import sparse_attention_paged_gb300 as lib
    ws = _fused_ws_floats(w.R, w.W, k)
    st2, i2, v2, s2 = _topk_form(w, k, lib.TOPK_TWO_PASS)
    stf, i_f, v_f, sf = _topk_form(w, k, lib.TOPK_FUSED, ws)
    assert st2 == 0 and stf == 0
    assert s2 == expect_status and sf == expect_status
    assert np.array_equal(i2, i_f)
    assert np.array_equal(v2.view(np.uint32), v_f.view(np.uint32))
    return i_f, v_f


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
@pytest.mark.parametrize("k", [1, 64, 300, 1024, 2048])
def test_topk_fused_matches_two_pass(kv, k):
    """Rows shorter than k, of exactly k, crossing several 2,048-position
    chunks, and the whole table; a ragged last page."""
    W = 150
    T = W * 64
    lens = [0, 1, 63, k, k + 1, 2047, 2048, 2049, 4100, 7000, T - 1, T]
    w = wl.decode_with_lengths(f"tkf{k}", lens, W, seed=60 + k, kv_dtype=kv)
    idx, val = _same_as_two_pass(w, k)
    _check(w, k, idx, val, list(range(w.R)))


def test_topk_many_rows_both_forms():
    """300 requests over a 70-page table: the two-pass selection runs one CTA
    per request (2 * B CTAs no longer fit in one wave), the fused form's
    slot header holds 300 rows; both forms agree bit for bit and the
    selection is a valid top-k of the oracle's logits."""
    g = np.random.default_rng(65)
    lens = [int(x) for x in g.integers(0, 70 * 64 + 1, 300)]
    lens[:5] = [0, 1, 64, 70 * 64, 130]
    k = 128
    w = wl.decode_with_lengths("tk_many", lens, 70, seed=65)
    idx, val = _same_as_two_pass(w, k)
    _check(w, k, idx, val, [0, 1, 2, 3, 4, 57, 150, 299])


def test_topk_fused_ties_bad_pages_and_long_rows():
    """Tied logits (an all-zero query, zeroed pages), a page id outside the
    pool (NaN logits, status 6) and an over-long row (status 7): both forms
    agree bit for bit and report the same status."""
    W, k = 120, 256
    lens = [5000, 5000, 3000, 7680, 7681, 900]
    w = wl.decode_with_lengths("tkf_ties", lens, W, seed=61)
    w.q_bits[0] = 0
    for pg in w.block_table[1, :20]:
        base = int(pg) * w.page_stride
        w.kcache[base: base + 8192] = 0
    w.block_table = w.block_table.copy()
    w.block_table[5, 3] = w.num_pages + 9
    _same_as_two_pass(w, k, expect_status=7)


def test_topk_fused_config3_batch():
    import sparse_attention_paged_gb300 as lib
    w = wl.cfg3(4097)
    for k in (256, 1000):
        idx, val = _same_as_two_pass(w, k)
        L = w.seqlens
        rows = sorted(set([int(np.argmin(L)), int(np.argmax(L)), 0, 1, 17, 63]))
        _check(w, k, idx, val, rows)
    # the contract's workspace (B * W * 64 floats) holds the fused form's
    # slots at k = 256, and the automatic form returns the same selection
    st, i_a, v_a, s = _topk_form(w, 256, lib.TOPK_AUTO)
    st_f, i_f, v_f, _ = _topk_form(w, 256, lib.TOPK_FUSED)
    assert st == 0 and st_f == 0 and s == 0
    assert np.array_equal(i_a, i_f)
    assert np.array_equal(v_a.view(np.uint32), v_f.view(np.uint32))


def test_topk_fused_refused_where_it_does_not_apply():
    import sparse_attention_paged_gb300 as lib
    # a short table (W <= 64) decodes per request: no fused form
    w = wl.decode_with_lengths("tkf_short", [100, 2000], 40, seed=62)
    st, idx, _, _ = _topk_form(w, 64, lib.TOPK_FUSED, _fused_ws_floats(2, 40, 64))
    assert st == 2 and (idx == -7).all()
    # k above a chunk
    w = wl.decode_with_lengths("tkf_bigk", [100, 9000], 150, seed=63)
    st, _, _, _ = _topk_form(w, 2049, lib.TOPK_FUSED, _fused_ws_floats(2, 150, 2049))
    assert st == 2
    # a workspace too small for the slots
    st, _, _, _ = _topk_form(w, 512, lib.TOPK_FUSED)
    assert st == 2
    # an unknown form
    st, _, _, _ = _topk_form(w, 64, 7)
    assert st == 1


def test_topk_fused_row_with_more_candidates_than_shared_memory():
    """Two requests over a 1,700-page table: the CTAs' slices are a few pages
    each, so every chunk keeps all of its positions and the long row's
    candidates (about 100,000) exceed what the merge stages in shared memory;
    it reads them in place instead."""
    W, k = 1700, 1024
    w = wl.decode_with_lengths("tkf_huge", [100000, 4000], W, seed=64)
    idx, val = _same_as_two_pass(w, k)
    _check(w, k, idx, val, [0, 1])
