"""GPU parity of the key-cache store: the library's bytes against the
oracle's, bit for bit (codes, scales and untouched slots), through the C
ABI; then the stored pages feed the indexer."""
import numpy as np
import pytest

import oracle
from sparse_attention_paged_gb300 import workloads as wl
from tests.parity import DeviceWorkload, compare, oracle_rows

pytestmark = pytest.mark.gpu


def _gpu_store(sw, out_pool=None):
    import torch
    import sparse_attention_paged_gb300 as lib
    k = torch.from_numpy(sw.k_bits.view(np.int16)).cuda()
    sl = torch.from_numpy(sw.slots).cuda()
    kc = torch.from_numpy(sw.kcache.copy()).cuda() if out_pool is None else out_pool
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = lib.dsa_kcache_store(k, sl, sw.n, kc, sw.page_stride, sw.num_pages, sw.kv_dtype,
                              128, 64, status)
    assert st == 0
    torch.cuda.synchronize()
    return kc, int(status.item())


def _oracle_store(sw):
    pool = sw.kcache.copy()
    st = oracle.kcache_store(sw.k_bits, sw.slots, pool, sw.page_stride, sw.num_pages, sw.kv_dtype)
    return pool, st


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_store_bytes_match_the_oracle(kv):
    sw = wl.store_rows("st", 3000, 60, seed=1, kv_dtype=kv, n_skip=40, n_bad=3)
    # rows the definition treats specially: all zero, signed zeros, values
    # that round to zero, one huge value
    k = sw.k_bits.copy()
    k[5] = 0
    k[6, :50] = 0x8000
    k[7, 3] = 0x3000                    # 2^-31: rounds to zero next to the row's other values
    k[8, 0] = 0x4F80                    # 2^32
    sw.k_bits = k
    kc, st = _gpu_store(sw)
    ref, st_ref = _oracle_store(sw)
    assert st == st_ref == oracle.BAD_PAGE
    got = kc.cpu().numpy()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"


def test_store_many_rows_fp8():
    sw = wl.store_rows("st_big", 20000, 400, seed=2)
    kc, st = _gpu_store(sw)
    ref, st_ref = _oracle_store(sw)
    assert st == st_ref == 0
    assert np.array_equal(kc.cpu().numpy(), ref)


def test_stored_pages_feed_the_indexer():
    """Keys stored by the library, read back by the decode kernel, against
    the oracle's logits over the oracle-stored pool (the same bytes)."""
    import torch
    W, B = 12, 6
    pool_pages = B * W
    sw = wl.store_rows("st_dec", pool_pages * 64, pool_pages, seed=3)
    sw.slots = np.arange(pool_pages * 64, dtype=np.int32)     # fill every slot
    kc, st = _gpu_store(sw)
    ref_pool, st_ref = _oracle_store(sw)
    assert st == st_ref == 0
    assert np.array_equal(kc.cpu().numpy(), ref_pool)
    g = np.random.default_rng(4)
    lens = g.integers(1, W * 64 + 1, B).astype(np.int32)
    bt = g.permutation(pool_pages).astype(np.int32).reshape(B, W)
    q = wl._bf16_bits(torch.from_numpy(g.normal(0, 1, (B, 64, 128)).astype(np.float32)))
    w = (g.normal(0, 1, (B, 64)) / 8).astype(np.float32)
    dec = wl.Workload(name="stored", kind="decode", kv_dtype=wl.KV_E4M3, R=B, W=W, q_bits=q, w=w,
                      kcache=ref_pool, page_stride=wl.FP8_PAGE_BYTES, num_pages=pool_pages,
                      kscale_offset=wl.FP8_SCALE_OFFSET, block_table=bt, bt_stride=W,
                      seqlens=lens)
    dw = DeviceWorkload(dec)
    assert dw.call() == 0
    torch.cuda.synchronize()
    assert int(dw.status.item()) == 0
    ref, st = oracle_rows(dec)
    assert st == 0
    compare(dw.out.cpu().numpy(), ref)
