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
            # one launch per group of up to 128 requests holding any row
            groups = [(b0, min(b0 + 128, len(cu) - 1)) for b0 in range(0, len(cu) - 1, 128)]
            assert n == sum(1 for a, b in groups if cu[b] > cu[a])
            assert c.host_table().shape == (len(cu) - 1, w.W)
        else:
            assert n == 1
        if w.kind != "store":
            assert c.host_table().shape[1] == w.W
        assert c.nbytes() > 0


def test_varlen_launch_count():
    """The varlen prefill launches once per group of up to 128 requests that
    holds any row: 4 requests -> 1, 131 -> 2, an empty group -> none."""
    class C:
        pass
    for cu, want in (([0, 5, 9, 9, 20], 1), (list(range(132)), 2),
                     ([0] * 129 + [1, 2, 3], 1), ([0, 0, 0], 0)):
        c = bench.DeviceCall.__new__(bench.DeviceCall)
        c.w = C()
        c.w.kind = "prefill"
        c.cu_q = cu
        assert c.launches() == want, (cu[:5], want)


def test_sweep_covers_every_configuration():
    """The per-configuration records name every configuration of the five
    (both calls of config 2, config 3 at both widths, the short lengths
    capped and uncapped)."""
    assert set(bench.SWEEP) <= set(wl.NAMED)
    assert {"1", "2a", "2b", "3", "3ref", "3short", "3short_capped", "4", "5"} == set(bench.SWEEP)
    for name in bench.SWEEP:
        assert len(wl.NAMED[name]()) == 1


def test_rotating_copies_exceed_twice_the_l2():
    for name in ("1", "2b", "3", "4"):
        works = wl.NAMED[name]()
        n = bench.n_copies_for(works)
        assert n * sum(w.algorithmic_bytes() for w in works) > 2 * bench.L2_BYTES


def test_stacked_copies_are_independent_views():
    torch = pytest.importorskip("torch")
    w = wl.cfg2b()
    copies = bench.make_copies([w], torch.device("cpu"), 3)
    ptrs = set()
    for cs in copies:
        c = cs[0]
        assert c.q.shape == (w.R, 64, 128) and c.out.shape == (w.R, w.W * 64)
        assert bool((c.seqlens.numpy() == w.seqlens).all())
        assert bytes(c.kcache.numpy()) == bytes(w.kcache)
        for t in (c.q, c.wt, c.kcache, c.bt, c.seqlens, c.out, c.status):
            assert t.data_ptr() % 16 == 0
            ptrs.add(t.data_ptr())
        assert c.kscale == c.kcache.data_ptr() + w.kscale_offset
    assert len(ptrs) == 3 * 7


def test_roofline_record_bounds():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1700.0}
    w4 = wl.cfg4()
    us = w4.algorithmic_bytes() / 6000e9 * 1e6 * 2          # half the HBM peak
    r = bench.roofline_record(w4, us, peaks)
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-9
    assert abs(r["t_roof_us"] - us / 2) < 1e-6
    w5 = wl.cfg5()
    us = w5.flops() / 2000e12 * 1e6 / 0.75
    r = bench.roofline_record(w5, us, peaks)
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.75) < 1e-9
    assert abs(r["frac_sustained"] - 0.75 * 2000 / 1700) < 1e-9


def test_config_record_carries_recorded_traffic():
    """A per-configuration record reports the ncu DRAM bytes recorded for
    its kernel, or None where none match the current sources."""
    w = wl.NAMED["3"]()[0]
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1700.0}
    rec = bench.config_record("3", w, 30.0, 100, 3.0, 4, 2**30, peaks, {})
    assert "traffic" in rec
    assert rec["traffic"] == bench.recorded_traffic(w.kind, w.name)
