"""Failure detection without a GPU fault: a bounded wait that runs out.

A test-only build of the library (compiled here into a temporary directory,
never shipped) leaves the first page tile of a CTA undelivered and shortens
every wait bound to ~10 ms.  The MMA warp's wait for that tile runs out; the
kernel must report DSA_ERR_TIMEOUT in the device status word, write NaN where
it could not compute a value, keep -inf where the length masks the position,
wait for its own copies in flight, free its TMEM and return -- after which
the context is still usable for a normal call.
"""
import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from sparse_attention_paged_gb300 import _native
from sparse_attention_paged_gb300 import workloads as wl
from tests.parity import DeviceWorkload, compare, oracle_rows

pytestmark = pytest.mark.gpu

TEST_FLAGS = ["-DDSA_TEST_SKIP_FIRST_TILE", "-DDSA_WAIT_LIMIT_CYCLES=20000000ll"]


def _build_variant(out_dir):
    def one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        subprocess.run([_native.NVCC, *_native.ARCH_FLAGS, *_native.NVCC_FLAGS, *TEST_FLAGS,
                        "-c", src, "-o", obj], check=True, capture_output=True)
        return obj
    srcs = _native._sources()
    with ThreadPoolExecutor(len(srcs)) as ex:
        objs = list(ex.map(one, srcs))
    lib = os.path.join(out_dir, "libdsa_indexer_timeout_test.so")
    subprocess.run([_native.NVCC, *_native.ARCH_FLAGS, "-shared", "-o", lib, *objs], check=True)
    L = ctypes.CDLL(lib)
    vp, ll, ci = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int
    L.dsa_indexer_logits_decode.restype = ci
    L.dsa_indexer_logits_decode.argtypes = [vp, vp, vp, vp, ll, ci, ci, vp, ll, vp, ci, ci, ci,
                                            ci, ci, vp, ll, vp, vp]
    return L


@pytest.mark.parametrize("kv", [wl.KV_E4M3, wl.KV_BF16])
def test_wait_that_runs_out_reports_timeout(tmp_path, kv):
    import torch
    torch.cuda.set_device(0)
    lib = _build_variant(str(tmp_path))
    L = 200
    w = wl.decode_with_lengths("timeout", [L], 4, seed=21, kv_dtype=kv)
    dw = DeviceWorkload(w)
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.dsa_indexer_logits_decode(
        dw.q.data_ptr(), dw.wt.data_ptr(), dw.kcache.data_ptr(), dw.kscale_ptr, w.page_stride,
        w.num_pages, w.kv_dtype, dw.bt.data_ptr(), w.bt_stride, dw.seqlens.data_ptr(), w.R,
        64, 128, 64, w.W, dw.out.data_ptr(), dw.out.stride(0), dw.status.data_ptr(), stream)
    assert st == 0
    torch.cuda.synchronize()                      # returns: the kernel did not hang
    assert int(dw.status.item()) == 5             # DSA_ERR_TIMEOUT
    o = dw.out.cpu().numpy()
    assert np.isnan(o[0, :L]).all()               # nothing computed is reported as a value
    assert np.isneginf(o[0, L:]).all()            # the mask still holds
    # the context is intact: a normal call through the product library works
    ok = DeviceWorkload(w)
    assert ok.call() == 0
    torch.cuda.synchronize()
    assert int(ok.status.item()) == 0
    compare(ok.out.cpu().numpy(), oracle_rows(w)[0])
