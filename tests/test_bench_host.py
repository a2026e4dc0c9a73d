"""bench.py's host-side bookkeeping for every named workload, on the CPU (the
call objects are built with CPU tensors; nothing is launched): every
workload has a description and a step count, and its call objects report
their kernel launches, table and sizes."""
import pytest

import bench
from sparse_attention_paged_gb300 import workloads as wl


def test_every_workload_is_described():
    assert set(bench.WORKLOAD_DESC) == set(wl.NAMED)
    assert set(bench.DEFAULT_STEPS) == set(wl.NAMED)


@pytest.mark.parametrize("name", sorted(wl.NAMED))
def test_call_objects(name):
    torch = pytest.importorskip("torch")
    for w in wl.NAMED[name]():
        c = bench.DeviceCall(w, torch.device("cpu"))
        n = c.launches()
        if w.kind == "topk":
            assert n == 2
        elif w.meta.get("varlen"):
            cu = c.cu_q
            assert cu[0] == 0 and cu[-1] == w.R
            assert n == sum(1 for a, b in zip(cu, cu[1:]) if b > a)
            assert c.host_table().shape == (len(cu) - 1, w.W)
        else:
            assert n == 1
        if w.kind != "store":
            assert c.host_table().shape[1] == w.W
        assert c.nbytes() > 0
