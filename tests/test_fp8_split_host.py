"""The fp8-key decode's query representation, emulated on the CPU.

For fp8 keys the decode kernel feeds the tensor cores the bf16 query as two
e4m3 terms under a per-head power of two 2^e (the head's largest |q| scaled
into [128, 256)): hi = e4m3(q 2^e) and lo = e4m3((q 2^e - hi) 2^5), the two
accumulated apart and joined as hi + lo 2^-5.  These tests emulate that
representation in float64 and show that the adversarial inputs of
test_gpu_parity's outlier / zero-key case separate it from the cheaper
single-accumulator split (lo = e4m3(q 2^e - hi), no 2^5), which misses the
1e-3 bar there.  The GPU test then checks the kernel itself on the same
inputs.
"""
import numpy as np
import pytest
import torch

from sparse_attention_paged_gb300 import workloads as wl

E4M3 = getattr(torch, "float8_e4m3fn", None)
pytestmark = pytest.mark.skipif(E4M3 is None, reason="torch without float8_e4m3fn")


def _scaled(q):
    m = q.abs().amax(-1, keepdim=True)
    E = torch.floor(torch.log2(m.clamp_min(1e-300)))
    e = torch.where(m > 0, (7 - E).clamp(-126, 126), torch.zeros_like(E))
    return q * torch.exp2(e), e


def _e4m3(x):
    return x.float().to(E4M3).double()


def split_one_accumulator(q):
    a, e = _scaled(q)
    hi = _e4m3(a)
    return (hi + _e4m3(a - hi)) * torch.exp2(-e)


def split_two_accumulators(q):
    a, e = _scaled(q)
    hi = _e4m3(a)
    r = (a - hi) * 32.0
    assert float(r.abs().max()) <= 448.0
    return (hi + _e4m3(r) / 32.0) * torch.exp2(-e)


def _dense_logits(w, qf):
    """Max |logit| and the logits of every valid position, computed densely
    with the query qf [R, H, D] (float64)."""
    pool = w.kcache.reshape(w.num_pages, w.page_stride)
    keys = torch.from_numpy(np.ascontiguousarray(pool[:, :wl.FP8_SCALE_OFFSET])).view(E4M3)
    keys = keys.double().reshape(w.num_pages, wl.P, wl.D)
    scale = torch.from_numpy(np.ascontiguousarray(pool[:, wl.FP8_SCALE_OFFSET:]).view(np.float32))
    wt = torch.from_numpy(w.w).double()
    out = []
    for r in range(w.R):
        L = int(w.seqlens[r])
        n = (L + wl.P - 1) // wl.P
        pages = torch.from_numpy(w.block_table[r, :n].astype(np.int64))
        k = keys[pages].reshape(-1, wl.D)[:L]
        s = scale[pages].double().reshape(-1)[:L]
        out.append(s * (torch.relu(k @ qf[r].T) @ wt[r]))
    return torch.cat(out)


def _case():
    w = wl.decode_uniform("wr_z", 16, 32, 2048, 512, seed=47)
    w.q_bits = wl.wide_range_queries(w.R, seed=54, outlier_d=5)
    wl.zero_key_dim(w, 5)
    q = torch.from_numpy(w.q_bits.view(np.int16)).view(torch.bfloat16).double()
    return w, q


def test_outlier_zero_key_case_separates_the_splits():
    w, q = _case()
    ref = _dense_logits(w, q)
    mref = float(ref.abs().max())
    assert mref > 0
    err_one = float((_dense_logits(w, split_one_accumulator(q)) - ref).abs().max()) / mref
    err_two = float((_dense_logits(w, split_two_accumulators(q)) - ref).abs().max()) / mref
    assert err_one > 1e-3, err_one
    assert err_two < 1e-5, err_two


def test_two_accumulator_split_is_exact_on_bf16_down_to_2_to_minus_15():
    """Every bf16 value at least 2^-14 of its head's largest comes back
    exactly; smaller ones within 2^-22 of the head's largest."""
    g = torch.Generator().manual_seed(3)
    big = torch.sign(torch.randn(4096, 1, generator=g, dtype=torch.float64)) * 2.0 ** \
        torch.randint(-20, 20, (4096, 1), generator=g).double()
    small = torch.randn(4096, 127, generator=g, dtype=torch.float64) * \
        2.0 ** (-20 * torch.rand(4096, 127, generator=g, dtype=torch.float64))
    q = torch.cat([big, small * big.abs()], 1).float().to(torch.bfloat16).double()
    got = split_two_accumulators(q)
    m = q.abs().amax(-1, keepdim=True)
    near = q.abs() >= m * 2.0 ** -14
    assert torch.equal(got[near], q[near])
    assert float(((got - q).abs() / m).max()) <= 2.0 ** -22
