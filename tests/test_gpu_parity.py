"""GPU parity: the CUDA library, called through its C ABI, against the fp64
oracle on the same seeded bytes.  The -inf mask must agree exactly and the
finite logits within max|d| <= 1e-3 * max|logit| (per call)."""
import numpy as np
import pytest

from sparse_attention_paged_gb300 import workloads as wl
from tests.parity import DeviceWorkload, compare, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    from sparse_attention_paged_gb300 import _native
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _native.build()
    yield


def _run(w, **kw):
    import torch
    dw = DeviceWorkload(w)
    st = dw.call(**kw)
    assert st == 0, st
    torch.cuda.synchronize()
    return dw


def _check_full(w):
    dw = _run(w)
    assert int(dw.status.item()) == 0
    ref, st = oracle_rows(w)
    assert st == 0
    return compare(dw.out.cpu().numpy(), ref)


# --- the small decode configurations, several seeds ----------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("shape", [(1, 8, 512, 16), (16, 32, 2048, 512), (32, 16, 1024, 512)],
                         ids=["B1_W8", "B16_W32", "B32_W16"])
def test_decode_fp8_small(shape, seed):
    B, W, Lmax, pool = shape
    _check_full(wl.decode_uniform(f"s{seed}", B, W, Lmax, pool, seed=seed))


def test_named_config_1_and_2():
    for w in [wl.cfg1(), wl.cfg2a(), wl.cfg2b()]:
        _check_full(w)


@pytest.mark.parametrize("idx", range(5))
def test_pages_validation_shapes(idx):
    _check_full(wl.pages_validation_cases()[idx])


@pytest.mark.parametrize("seed", [0, 1])
def test_decode_bf16_small(seed):
    _check_full(wl.decode_uniform(f"bf{seed}", 8, 12, 12 * 64, 200, seed=seed,
                                  kv_dtype=wl.KV_BF16))


# --- edges ------------------------------------------------------------------

@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_edge_lengths(kv):
    W = 5
    T = W * 64
    lengths = [0, 1, 63, 64, 65, 127, 128, 129, T - 1, T, -3, 200]
    _check_full(wl.decode_with_lengths("edges", lengths, W, seed=3, kv_dtype=kv))


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_single_page_table(kv):
    _check_full(wl.decode_with_lengths("w1", [1, 17, 64, 0, 33], 1, seed=4, kv_dtype=kv))


def test_zero_rows_is_a_no_op():
    import torch
    import sparse_attention_paged_gb300 as lib
    w = wl.cfg1()
    dw = DeviceWorkload(w)
    dw.out.fill_(7.0)
    st = lib.dsa_indexer_logits_decode(dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w.page_stride,
                                       w.num_pages, w.kv_dtype, dw.bt, w.bt_stride, dw.seqlens,
                                       0, 64, 128, 64, w.W, dw.out, dw.out.stride(0), None, None)
    torch.cuda.synchronize()
    assert st == 0 and bool((dw.out == 7.0).all())


def test_strided_output_and_table():
    """out_stride > W*64 and bt_stride > W: padding is left untouched."""
    import torch
    w = wl.decode_uniform("strided", 6, 7, 7 * 64, 64, seed=9)
    ref, _ = oracle_rows(w)
    dw = DeviceWorkload(w)
    bt_wide = torch.full((w.R, w.W + 3), -5, dtype=torch.int32, device="cuda")
    bt_wide[:, : w.W] = dw.bt
    out_wide = torch.full((w.R, w.W * 64 + 36), 3.0, device="cuda")
    import sparse_attention_paged_gb300 as lib
    st = lib.dsa_indexer_logits_decode(dw.q, dw.wt, dw.kcache, dw.kscale_ptr, w.page_stride,
                                       w.num_pages, w.kv_dtype, bt_wide, w.W + 3, dw.seqlens,
                                       w.R, 64, 128, 64, w.W, out_wide, out_wide.stride(0),
                                       dw.status, None)
    torch.cuda.synchronize()
    assert st == 0
    o = out_wide.cpu().numpy()
    compare(o[:, : w.W * 64], ref)
    assert (o[:, w.W * 64:] == 3.0).all()


# --- data errors: reported in-kernel, never a fault --------------------------

def test_bad_page_id_poisons_its_positions():
    import torch
    w = wl.decode_with_lengths("badpage", [150, 70], 3, seed=5)
    w.block_table = w.block_table.copy()
    w.block_table[0, 1] = w.num_pages + 11        # needed by row 0 (positions 64..127)
    w.block_table[1, 2] = -4                      # not needed by row 1 (L = 70)
    dw = _run(w)
    assert int(dw.status.item()) == 6
    ref, st = oracle_rows(w)
    assert st == 6
    compare(dw.out.cpu().numpy(), ref)


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_balanced_bad_page_ids(kv):
    """Long tables (the balanced split): every fifth table entry of two rows
    lies outside the pool (some are the first page of a CTA's slice, whose
    entries the fp8 path reads ahead) and one is negative; their positions
    are NaN, the call reports status 6, and every other position is
    exact."""
    W = 90
    w = wl.decode_with_lengths("bal_badpage", [5000, 3000, W * 64, 700, 64], W, seed=71,
                               kv_dtype=kv)
    w.block_table = w.block_table.copy()
    w.block_table[0, ::5] = w.num_pages + 3
    w.block_table[2, 2::5] = w.num_pages + 100
    w.block_table[3, 4] = -1
    dw = _run(w)
    assert int(dw.status.item()) == 6
    ref, st = oracle_rows(w)
    assert st == 6
    compare(dw.out.cpu().numpy(), ref)


def test_length_past_table_is_a_nan_row():
    w = wl.decode_with_lengths("badlen", [100, 3 * 64 + 1, 5], 3, seed=6)
    dw = _run(w)
    assert int(dw.status.item()) == 7
    ref, st = oracle_rows(w)
    assert st == 7
    o = dw.out.cpu().numpy()
    assert np.isnan(o[1]).all()
    compare(o, ref)


@pytest.mark.parametrize("kv,W,lengths", [
    (wl.KV_E4M3, 90, [5000, 90 * 64 + 1, 3000, 0, 90 * 64, 64, 65]),
    (wl.KV_BF16, 2048, [2048 * 64, 2048 * 64 + 1, 100000, 70000, 2048 * 64]),
], ids=["fp8_fill_lanes", "bf16_paced_fill"])
def test_balanced_length_past_table_is_a_nan_row(kv, W, lengths):
    """Long tables (the balanced split) with a row longer than the table:
    that whole row is NaN, written by the fill's bulk copies from the NaN
    block, and the call reports status 7; every other row is exact.  The
    bf16 case holds about 22 pages per CTA, so its fill goes out paced from
    the producer's lane 0; the fp8 case goes through the 31 fill lanes."""
    w = wl.decode_with_lengths(f"bal_badlen_{W}", lengths, W, seed=70, kv_dtype=kv)
    dw = _run(w)
    assert int(dw.status.item()) == 7
    ref, st = oracle_rows(w)
    assert st == 7
    o = dw.out.cpu().numpy()
    assert np.isnan(o[1]).all()
    compare(o, ref)


# --- CUDA graph capture: fixed grid, data-dependent work --------------------

def test_graph_capture_and_replay_with_new_lengths():
    import torch
    w0 = wl.decode_uniform("g0", 16, 32, 2048, 512, seed=0)
    w1 = wl.decode_uniform("g1", 16, 32, 2048, 512, seed=1)
    dw = DeviceWorkload(w0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dw.call()                                   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = dw.call()
    assert st == 0
    g.replay()
    torch.cuda.synchronize()
    compare(dw.out.cpu().numpy(), oracle_rows(w0)[0])
    # new inputs in the same buffers: lengths, table, q, w and cache all change
    dw.q.copy_(DeviceWorkload(w1).q)
    for name in ("wt", "kcache", "bt", "seqlens"):
        getattr(dw, name).copy_(getattr(DeviceWorkload(w1), name))
    g.replay()
    torch.cuda.synchronize()
    compare(dw.out.cpu().numpy(), oracle_rows(w1)[0])


# --- full-size configurations ------------------------------------------------

@pytest.mark.parametrize("W", [4097, 512])
def test_config3_full(W):
    stats = _check_full(wl.cfg3(W))
    assert stats["rel"] < 1e-3


@pytest.mark.parametrize("W", [4097, 32])
def test_config3_short_lengths_capped_and_uncapped(W):
    _check_full(wl.cfg3_short(W))


def test_config3_width_does_not_change_valid_logits():
    """Same lengths, width 4097 vs 512: identical values below each length
    (the table's extra entries are never read)."""
    a = _run(wl.cfg3(4097)).out.cpu().numpy()
    b = _run(wl.cfg3(512)).out.cpu().numpy()
    assert np.array_equal(a[:, : 512 * 64], b)
    assert np.isneginf(a[:, 512 * 64:]).all()


def _sampled(w, rows):
    dw = _run(w)
    assert int(dw.status.item()) == 0
    o = dw.out.cpu().numpy()
    # mask and NaN-freedom on every row, values on the sampled rows
    T = w.W * w.P
    L = np.clip(w.seqlens.astype(np.int64), 0, T)
    assert np.array_equal(np.isneginf(o), np.arange(T)[None, :] >= L[:, None])
    assert not np.isnan(o).any()
    ref, st = oracle_rows(w, rows)
    assert st == 0
    return compare(o[rows], ref)


def test_config4_bf16_full_size_all_rows():
    """All 64 requests of the bf16 decode configuration, every position."""
    stats = _check_full(wl.cfg4())
    assert stats["rel"] < 1e-3


def config5_rows(n_sms: int) -> list[int]:
    """Rows of the full-size prefill to compare value by value: the first
    and the last query of every 8th query tile, and of the query tiles
    where each persistent CTA's slice of the (query tile, position tile)
    item list starts and ends.  The kernel gives each of its n_sms CTAs an
    equal share of the list's cost (an item weighs 16, a query tile adds 32
    and 1/20 per page of its rows' tail past its last position tile); CTA k
    starts at the first item whose cost range begins at or after k/n_sms of
    the total, which is recomputed here."""
    w = wl.cfg5()
    T = w.W * w.P
    L = np.where(w.seqlens > T, 0, np.clip(w.seqlens, 0, T)).astype(np.int64)
    n_qt = (w.R + 3) // 4
    lmax = np.array([L[4 * j: 4 * j + 4].max() for j in range(n_qt)])
    nrow = np.array([min(4, w.R - 4 * j) for j in range(n_qt)])
    nt = (lmax + 127) // 128
    wt = np.where(nt > 0, 16 * nt + 32 + nrow * np.maximum(w.W - 2 * nt, 0) // 20, 0)
    cum = np.concatenate([[0], np.cumsum(wt)])
    total = int(cum[-1])

    def tile_rows(j):
        return (4 * j, min(4 * j + 3, w.R - 1))

    rows = set()
    for j in range(0, n_qt, 8):
        rows.update(tile_rows(j))
    for k in range(1, n_sms):
        x = k * total // n_sms
        j = int(np.searchsorted(cum, x, side="right") - 1)
        if j >= n_qt:
            continue
        rows.update(tile_rows(j))          # the CTA's first item is in tile j ...
        if j > 0:
            rows.update(tile_rows(j - 1))  # ... or is tile j's first, the previous CTA ending in j - 1
    rows.update((0, w.R - 1))
    return sorted(rows)


def test_config5_prefill_full_size_sampled_rows():
    import torch
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = config5_rows(n_sms)
    assert len(rows) >= 512
    _sampled(wl.cfg5(), rows)


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_E4M3])
def test_prefill_small_full(kv):
    # 70 queries: 18 query tiles, the last one ragged
    _check_full(wl.prefill_causal("pf_small", 70, 9, 9 * 64 - 75, seed=2, kv_dtype=kv))


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_E4M3])
def test_prefill_bad_page_id(kv):
    w = wl.prefill_causal("pf_badpage", 30, 6, 6 * 64 - 40, seed=9, kv_dtype=kv)
    w.block_table = w.block_table.copy()
    w.block_table[0, 2] = w.num_pages + 3          # positions 128..191, needed by every query
    dw = _run(w)
    assert int(dw.status.item()) == 6
    ref, st = oracle_rows(w)
    assert st == 6
    compare(dw.out.cpu().numpy(), ref)


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_E4M3])
def test_prefill_length_past_table(kv):
    w = wl.prefill_causal("pf_badlen", 30, 6, 6 * 64 - 40, seed=10, kv_dtype=kv)
    w.seqlens = w.seqlens.copy()
    w.seqlens[5] = w.W * 64 + 1
    dw = _run(w)
    assert int(dw.status.item()) == 7
    ref, st = oracle_rows(w)
    assert st == 7
    o = dw.out.cpu().numpy()
    assert np.isnan(o[5]).all()
    compare(o, ref)


# --- prefill with per-query table rows (several requests in one call) and
# with fp8 keys: one decode row per query token ------------------------------

@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_E4M3])
def test_prefill_per_query_tables_small_full(kv):
    w = wl.prefill_varlen("pf_varlen", [(20, 150), (33, 400), (7, 64), (1, 1)], seed=3, kv_dtype=kv)
    assert w.bt_stride == w.W
    _check_full(w)


def test_prefill_fp8_shared_table_small_full():
    _check_full(wl.prefill_causal("pf_fp8", 60, 7, 7 * 64 - 70, seed=4, kv_dtype=wl.KV_E4M3))


def test_prefill_fp8_many_query_tiles():
    # several query tiles per CTA: the query split runs at every tile change
    _check_full(wl.prefill_causal("pf_fp8_many", 1200, 20, 50, seed=11, kv_dtype=wl.KV_E4M3))


def test_config6_varlen_prefill_sampled_rows():
    w = wl.cfg6()
    rows = []
    for a, n in w.meta["groups"]:            # first, middle and last token of every request
        rows += [a, a + n // 2, a + n - 1]
    _sampled(w, sorted(rows))


def test_config7_fp8_prefill_sampled_rows():
    _sampled(wl.cfg7(), [0, 1, 511, 512, 1022, 1023])


# --- launches overlap their prologue with the previous kernel (programmatic
# dependent launch): inputs written just before, and outputs written twice
# back to back, must still be ordered -----------------------------------------

def test_inputs_written_by_the_previous_kernel():
    import torch
    w0 = wl.decode_uniform("pdl0", 16, 32, 2048, 512, seed=0)
    w1 = wl.decode_uniform("pdl1", 16, 32, 2048, 512, seed=1)
    dw = DeviceWorkload(w0)
    src = DeviceWorkload(w1)
    torch.cuda.synchronize()
    for _ in range(3):
        # overwrite every input with a device kernel, then call immediately
        dw.q.copy_(src.q)
        dw.wt.copy_(src.wt)
        dw.kcache.copy_(src.kcache)
        dw.bt.copy_(src.bt)
        dw.seqlens.copy_(src.seqlens)
        assert dw.call() == 0
        out1 = dw.out.clone()
        dw.q.copy_(DeviceWorkload(w0).q)
        dw.wt.copy_(DeviceWorkload(w0).wt)
        dw.kcache.copy_(DeviceWorkload(w0).kcache)
        dw.bt.copy_(DeviceWorkload(w0).bt)
        dw.seqlens.copy_(DeviceWorkload(w0).seqlens)
        assert dw.call() == 0
    torch.cuda.synchronize()
    compare(out1.cpu().numpy(), oracle_rows(w1)[0])
    compare(dw.out.cpu().numpy(), oracle_rows(w0)[0])


@pytest.mark.parametrize("kind", ["decode", "prefill", "prefill_fp8"])
def test_back_to_back_calls_into_one_output(kind):
    """Two calls in a row write the same output buffer; the second's
    lengths are shorter, so any write of the first landing late would
    leave a finite value where the second wants -inf."""
    import torch
    if kind == "decode":
        a = wl.decode_with_lengths("bb_a", [2000, 1500, 900, 64], 32, seed=7)
        b = wl.decode_with_lengths("bb_b", [5, 70, 1, 0], 32, seed=7)
    else:
        kv = wl.KV_E4M3 if kind == "prefill_fp8" else wl.KV_BF16
        a = wl.prefill_causal("bb_a", 40, 12, 12 * 64 - 41, seed=8, kv_dtype=kv)
        b = wl.prefill_causal("bb_b", 40, 12, 100, seed=8, kv_dtype=kv)
    da, db = DeviceWorkload(a), DeviceWorkload(b)
    out = torch.empty_like(da.out)
    for _ in range(5):
        assert da.call(out=out) == 0
        assert db.call(out=out) == 0
    torch.cuda.synchronize()
    compare(out.cpu().numpy(), oracle_rows(b)[0])


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_more_ctas_than_sms_with_idle_ctas(kv):
    """Per-request mode with more CTAs than SMs (64 rows of a 32-page table:
    four CTAs a row, so the CTAs take their tensor memory before waiting for
    the previous launch) and rows short enough that some CTAs have no page
    and leave early; two calls back to back into one output, so that each
    launch's CTAs start while the previous launch runs."""
    import torch
    g = np.random.default_rng(21)
    lengths = [int(x) for x in g.integers(0, 32 * 64 + 1, 64)]
    lengths[:8] = [0, 1, 63, 64, 65, 127, 2048, -3]
    a = wl.decode_with_lengths("early_a", lengths, 32, seed=21, kv_dtype=kv)
    b = wl.decode_with_lengths("early_b", [max(0, x // 3) for x in lengths], 32, seed=21,
                               kv_dtype=kv)
    _check_full(a)
    da, db = DeviceWorkload(a), DeviceWorkload(b)
    out = torch.empty_like(da.out)
    for _ in range(3):
        assert da.call(out=out) == 0
        assert db.call(out=out) == 0
    torch.cuda.synchronize()
    compare(out.cpu().numpy(), oracle_rows(b)[0])


def test_concurrent_calls_on_three_streams():
    """Three calls issued repeatedly on three streams at once: an fp8 and a
    bf16 decode over long tables (two CTAs per SM each, tensor memory taken
    before the dependent-launch wait, so CTAs of different calls share SMs)
    and a per-request fp8 decode; every output stays exact."""
    import torch
    a = wl.decode_with_lengths("cc_a", [4400, 3000, 70 * 64, 100], 70, seed=80)
    b = wl.decode_with_lengths("cc_b", [4000, 64, 1, 70 * 64], 70, seed=81, kv_dtype=wl.KV_BF16)
    c = wl.decode_uniform("cc_c", 32, 16, 1024, 512, seed=82)
    ds = [DeviceWorkload(x) for x in (a, b, c)]
    streams = [torch.cuda.Stream() for _ in ds]
    torch.cuda.synchronize()
    for _ in range(20):
        for d, st in zip(ds, streams):
            assert d.call(stream=st.cuda_stream) == 0
    torch.cuda.synchronize()
    for x, d in zip((a, b, c), ds):
        assert int(d.status.item()) == 0
        compare(d.out.cpu().numpy(), oracle_rows(x)[0])


# --- long tables: CTAs are dispatched longest row first -----------------------

@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_longest_first_order_with_ties(kv):
    W = 70
    lengths = [500, 4000, 500, 4000, 0, W * 64, 1, 4000, -2, 64]
    _check_full(wl.decode_with_lengths("ties", lengths, W, seed=12, kv_dtype=kv))


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_balanced_with_the_most_rows(kv):
    """384 rows over a 65-page table, the most rows the balanced split takes
    (its per-row prefix sums live in shared memory): twelve 32-row chunks in
    the prefix sums and the slice search, rows of every length."""
    g = np.random.default_rng(14)
    lengths = g.integers(0, 65 * 64 + 1, 384)
    lengths[:6] = [0, 1, 64, 65, 65 * 64, 2]
    _check_full(wl.decode_with_lengths("most_rows", lengths, 65, seed=14, kv_dtype=kv))


def test_many_rows_long_table_natural_order():
    """More rows than the longest-first ordering handles: natural order."""
    g = np.random.default_rng(13)
    lengths = g.integers(0, 65 * 64 + 1, 400)
    _check_full(wl.decode_with_lengths("many", lengths, 65, seed=13))


# --- queries with a wide dynamic range per head: the fp8 path represents the
# bf16 query as two e4m3 terms under a per-head power-of-two scale; elements
# far below their head's largest are where that representation is least
# exact ----------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1])
def test_decode_fp8_wide_range_queries(seed):
    for w in (wl.decode_uniform(f"wr{seed}", 16, 32, 2048, 512, seed=40 + seed),
              wl.decode_with_lengths(f"wrl{seed}", [0, 1, 64, 65, 3000, 90 * 64],
                                     90, seed=42 + seed)):
        w.q_bits = wl.wide_range_queries(w.R, seed=50 + seed)
        stats = _check_full(w)
        assert stats["rel"] < 1e-3


def test_decode_fp8_outliers_meet_zero_keys():
    """Every head's outlier element sits at d = 5, where every key is zero,
    so the dots come from the heads' small elements alone: the inputs on
    which a query split with few bits below the head's largest element
    misses the bar (test_fp8_split_host shows one that does)."""
    for w in (wl.decode_uniform("wr_z", 16, 32, 2048, 512, seed=47),
              wl.decode_with_lengths("wrl_z", [1, 64, 3000, 90 * 64], 90, seed=48)):
        w.q_bits = wl.wide_range_queries(w.R, seed=54, outlier_d=5)
        wl.zero_key_dim(w, 5)
        stats = _check_full(w)
        assert stats["rel"] < 1e-4


def test_prefill_fp8_wide_range_queries():
    w = wl.prefill_causal("pf_wr", 130, 10, 10 * 64 - 140, seed=43, kv_dtype=wl.KV_E4M3)
    w.q_bits = wl.wide_range_queries(w.R, seed=52)
    _check_full(w)


def test_prefill_and_decode_bf16_wide_range_queries():
    for w in (wl.prefill_causal("pf_wr_bf", 70, 9, 9 * 64 - 75, seed=44),
              wl.decode_uniform("wr_bf", 8, 12, 12 * 64, 200, seed=45, kv_dtype=wl.KV_BF16)):
        w.q_bits = wl.wide_range_queries(w.R, seed=53)
        _check_full(w)


@pytest.mark.parametrize("kv", [wl.KV_BF16, wl.KV_E4M3])
@pytest.mark.parametrize("exp", [-40, 30])
def test_prefill_tiny_and_large_dots(kv, exp):
    """Queries scaled by 2^-40 (per-head dots near 2^-37) and by 2^30 (dots
    near 2^33): half of the heads take their ReLU as a saturating multiply
    by 2^-64, whose products must stay normal floats at the small end and
    below 1 at the large end."""
    import torch
    w = wl.prefill_causal(f"pf_sc{exp}", 40, 6, 6 * 64 - 50, seed=46, kv_dtype=kv)
    q = torch.from_numpy(w.q_bits.view(np.int16)).view(torch.bfloat16).float() * (2.0 ** exp)
    w.q_bits = q.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    stats = _check_full(w)
    assert stats["max_ref"] > 0
