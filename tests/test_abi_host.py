"""The C ABI on the host (no GPU needed): the library builds for sm_103a,
loads, exports every function include/dsa_indexer.h declares, and rejects
bad arguments before launching anything."""
import os
import re
import shutil

import pytest

from sparse_attention_paged_gb300 import _native

HEADER = os.path.join(_native.INCLUDE, "dsa_indexer.h")

needs_nvcc = pytest.mark.skipif(shutil.which(_native.NVCC) is None and
                                not os.path.exists(_native.LIB_PATH),
                                reason="nvcc not available and library not built")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _native.load()


@needs_nvcc
def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_native.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


@needs_nvcc
def test_abi_version_and_status_strings(lib):
    import sparse_attention_paged_gb300 as s
    assert s.dsa_indexer_abi_version() == 1
    for code, name in s.STATUS.items():
        assert s.dsa_status_string(code).startswith(name)
    assert "unknown" in s.dsa_status_string(99)


# Fake, suitably aligned device addresses: every call below must fail its
# host-side checks, so nothing is dereferenced or launched.
A = 0x10000


def call(fn="decode", **kw):
    import sparse_attention_paged_gb300 as s
    args = dict(q=A, w=A, kcache=A, kscale=A + 8192, page_stride_bytes=8448, num_pages=16,
                kv_dtype=0, block_table=A, bt_stride=8, seqlens=A, B=1, H=64, D=128,
                page_size=64, W=8, out=A, out_stride=512, dev_status=None, stream=0)
    args.update(kw)
    if fn == "prefill":
        args["n_q"] = args.pop("B")
        return s.dsa_indexer_logits_prefill(**args)
    return s.dsa_indexer_logits_decode(**args)


@needs_nvcc
@pytest.mark.parametrize("kw,code", [
    (dict(H=32), 2), (dict(D=64), 2), (dict(page_size=32), 2),
    (dict(W=0), 1), (dict(B=-1), 1), (dict(kv_dtype=2), 1),
    (dict(q=None), 1), (dict(out=None), 1), (dict(block_table=None), 1),
    (dict(seqlens=None), 1), (dict(w=None), 1), (dict(kcache=None), 1),
    (dict(num_pages=0), 1), (dict(page_stride_bytes=4096), 1),
    (dict(bt_stride=3), 1), (dict(out_stride=100), 1),
    (dict(page_stride_bytes=8456), 3), (dict(out_stride=514), 3),
    (dict(q=A + 8), 3), (dict(kcache=A + 4), 3), (dict(out=A + 4), 3),
    (dict(kscale=A + 8196), 3),
    (dict(kv_dtype=1, page_stride_bytes=8448), 1),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert call(**kw) == code


@needs_nvcc
def test_zero_rows_returns_ok_without_launch(lib):
    assert call(B=0) == 0


@needs_nvcc
def test_prefill_mode_checks(lib):
    # per-query table rows run one decode row per query token, whose grid
    # caps n_q at 65535; the checks come before any launch
    assert call("prefill", kv_dtype=0, bt_stride=8, B=70000) == 2             # fp8, per-query rows
    assert call("prefill", kv_dtype=1, page_stride_bytes=16384, kscale=None,
                bt_stride=8, B=70000) == 2                                    # per-query tables
    assert call("prefill", kv_dtype=1, page_stride_bytes=16384, kscale=None,
                bt_stride=0, B=0) == 0


def store_call(**kw):
    import sparse_attention_paged_gb300 as s
    args = dict(k=A, slot_mapping=A, n=4, kcache=A, page_stride_bytes=8448, num_pages=16,
                kv_dtype=0, D=128, page_size=64, dev_status=None, stream=0)
    args.update(kw)
    return s.dsa_kcache_store(**args)


@needs_nvcc
@pytest.mark.parametrize("kw,code", [
    (dict(D=64), 2), (dict(page_size=32), 2), (dict(kv_dtype=3), 1), (dict(n=-1), 1),
    (dict(num_pages=0), 1), (dict(k=None), 1), (dict(kcache=None), 1),
    (dict(slot_mapping=None), 1),
    (dict(page_stride_bytes=8192), 1),                    # fp8 pages need room for the scales
    (dict(kv_dtype=1, page_stride_bytes=8448), 1),        # bf16 pages hold 16 KB of values
    (dict(page_stride_bytes=8456), 3), (dict(k=A + 8), 3), (dict(kcache=A + 4), 3),
    (dict(slot_mapping=A + 2), 3),
])
def test_store_rejects_bad_arguments(lib, kw, code):
    assert store_call(**kw) == code


@needs_nvcc
def test_store_zero_rows_is_a_no_op(lib):
    assert store_call(n=0) == 0


def topk_call(**kw):
    import sparse_attention_paged_gb300 as s
    args = dict(q=A, w=A, kcache=A, kscale=A + 8192, page_stride_bytes=8448, num_pages=16,
                kv_dtype=0, block_table=A, bt_stride=8, seqlens=A, B=2, H=64, D=128,
                page_size=64, W=8, k_top=64, topk_idx=A, topk_val=A, topk_stride=64,
                workspace=A, workspace_floats=2 * 8 * 64, dev_status=None, stream=0)
    args.update(kw)
    return s.dsa_indexer_topk_decode(**args)


@needs_nvcc
@pytest.mark.parametrize("kw,code", [
    (dict(k_top=0), 1), (dict(topk_idx=None), 1), (dict(topk_stride=63), 1),
    (dict(workspace_floats=2 * 8 * 64 - 1), 1), (dict(workspace=None), 1),
    (dict(topk_idx=A + 2), 3), (dict(topk_val=A + 1), 3), (dict(workspace=A + 4), 3),
    (dict(H=32), 2), (dict(B=70000, workspace_floats=70000 * 512), 2),
])
def test_topk_rejects_bad_arguments(lib, kw, code):
    assert topk_call(**kw) == code


@needs_nvcc
def test_topk_zero_rows_is_a_no_op(lib):
    assert topk_call(B=0) == 0


def call_varlen(**kw):
    import sparse_attention_paged_gb300 as s
    args = dict(q=A, w=A, kcache=A, kscale=A + 8192, page_stride_bytes=8448, num_pages=16,
                kv_dtype=0, block_table=A, bt_stride=8, cu_q=[0, 3, 5], seqlens=A, H=64,
                D=128, page_size=64, W=8, out=A, out_stride=512, dev_status=None, stream=0)
    args.update(kw)
    return s.dsa_indexer_logits_prefill_varlen(**args)


@needs_nvcc
@pytest.mark.parametrize("kw, code", [
    (dict(cu_q=[1, 3, 5]), 1),                 # offsets must start at 0
    (dict(cu_q=[0, 5, 3]), 1),                 # and not decrease
    (dict(bt_stride=4), 1),                    # a table row per request: bt_stride >= W
    (dict(q=None), 1),
    (dict(H=32), 2),
    (dict(out_stride=256), 1),
    (dict(q=A + 8), 3),
])
def test_prefill_varlen_rejects_bad_arguments(lib, kw, code):
    assert call_varlen(**kw) == code


@needs_nvcc
def test_prefill_varlen_without_query_tokens_is_a_no_op(lib):
    # no rows: nothing is launched, whatever the (fake) pointers
    assert call_varlen(cu_q=[]) == 0
    assert call_varlen(cu_q=[0]) == 0
    assert call_varlen(cu_q=[0, 0, 0]) == 0
