"""Pins of the oracle's key-cache store (CPU only).

The store writes new key rows into their cache slots: the page layouts are
those the indexer reads ("The Dispatch Wire: Connecting a Triton Indexer
Kernel to Production Inference", section "The Reasoning and Decision-Making":
P*D e4m3 bytes followed by P fp32 scales; "The Dispatch Decision: Wiring a
Triton Kernel into Production", section "The Problem That Led Here": bf16
rows, no quantisation).  The quantisation rule is a reading (the pages give
none): s = max|k| / 448 in fp32, code = nearest e4m3 of k / s (fp32), ties to
even, saturated to +-448.  The e4m3 format is OCP FP8 E4M3 ("E4M3FN").

The expected codes below are worked out by hand from the format definition.
"""
import numpy as np
import pytest

import oracle

E4M3_MAX_CODE = 0x7E


def _bf16(x) -> np.ndarray:
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_every_finite_code_round_trips():
    for c in range(256):
        if c & 0x7F == 0x7F:          # the two NaN codes
            continue
        v = oracle.e4m3_to_double(c)
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_midpoints_round_to_the_even_code():
    vals = [oracle.e4m3_to_double(c) for c in range(0, E4M3_MAX_CODE + 1)]
    for c in range(E4M3_MAX_CODE):
        m = (vals[c] + vals[c + 1]) / 2           # exact in fp32: at most 5 significant bits
        assert np.float32(m) == m
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(m) == even, (c, m)
        assert oracle.e4m3_encode(-m) == 0x80 | even


def test_saturation_and_signed_zero():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(479.9) == 0x7E      # would round to 480, which is the NaN code
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-2.0 ** -11) == 0x80  # rounds to zero, keeps the sign
    assert oracle.e4m3_encode(2.0 ** -9) == 0x01    # the smallest subnormal


def test_encoder_matches_the_library_cast():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(3)
    x = np.concatenate([g.uniform(-448, 448, 4000), g.normal(0, 1, 4000),
                        g.normal(0, 0.01, 2000)]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(ours, lib)


def _pool(num_pages, D, P, fp8, fill=0xA5):
    stride = P * (D + 4) if fp8 else P * D * 2
    return np.full(num_pages * stride, fill, dtype=np.uint8), stride


def test_hand_rows_fp8():
    D, P = 4, 2
    pool, stride = _pool(2, D, P, fp8=True)
    k = np.stack([
        _bf16([448.0, 1.0, -3.0, 0.0]),          # s = 1: 448 -> 0x7E, 1 -> 0x38, -3 -> 0xC4, 0 -> 0x00
        _bf16([2.0, -0.5, 0.25, 1.75]),          # s = 2/448: 448 -> 0x7E, -112 -> 0xEE, 56 -> 0x66,
                                                 #   392 -> 384 (nearest) -> 0x7C
        _bf16([448.0, 17.0, 19.0, -2.0 ** -10]),  # ties: 17 -> 16 (0x58), 19 -> 20 (0x5A),
                                                 #   -2^-10 -> -0 (0x80)
        _bf16([0.0, 0.0, 0.0, 0.0]),             # all zero: s = 1, codes 0 (skipped below)
        _bf16([1.0, 1.0, 1.0, 1.0]),             # slot past the pool: skipped, status 6
    ])
    slots = np.array([3, 0, 2, -1, 4], dtype=np.int32)   # page 1 slot 1, page 0 slot 0, page 1 slot 0
    st = oracle.kcache_store(k, slots, pool, stride, 2, oracle.KV_E4M3, D=D, P=P)
    assert st == oracle.BAD_PAGE

    def codes(page, slot):
        return list(pool[page * stride + slot * D: page * stride + slot * D + D])

    def scale(page, slot):
        off = page * stride + P * D + slot * 4
        return pool[off: off + 4].view(np.float32)[0]

    assert codes(1, 1) == [0x7E, 0x38, 0xC4, 0x00] and scale(1, 1) == np.float32(1.0)
    assert codes(0, 0) == [0x7E, 0xEE, 0x66, 0x7C]
    assert scale(0, 0) == np.float32(2.0) / np.float32(448.0)
    assert codes(1, 0) == [0x7E, 0x58, 0x5A, 0x80] and scale(1, 0) == np.float32(1.0)
    # page 0 slot 1 was not written
    assert codes(0, 1) == [0xA5] * 4


def test_all_zero_row_has_scale_one():
    D, P = 4, 2
    pool, stride = _pool(1, D, P, fp8=True)
    st = oracle.kcache_store(_bf16([[0.0, -0.0, 0.0, 0.0]]), np.array([1], np.int32), pool,
                             stride, 1, oracle.KV_E4M3, D=D, P=P)
    assert st == 0
    assert list(pool[D: 2 * D]) == [0x00, 0x80, 0x00, 0x00]
    assert pool[P * D + 4: P * D + 8].view(np.float32)[0] == np.float32(1.0)


def test_bf16_rows_are_copied():
    D, P = 4, 2
    pool, stride = _pool(2, D, P, fp8=False)
    k = _bf16([[1.5, -2.0, 3.25, 0.0], [7.0, 8.0, 9.0, -10.0]])
    st = oracle.kcache_store(k, np.array([2, 1], np.int32), pool, stride, 2, oracle.KV_BF16,
                             D=D, P=P)
    assert st == 0
    assert np.array_equal(pool[stride: stride + 2 * D].view(np.uint16), k[0])
    assert np.array_equal(pool[2 * D: 4 * D].view(np.uint16), k[1])


def test_dequantised_error_bound():
    # |code * s - k| <= half a unit in the last place of e4m3 (3 mantissa
    # bits: 2^-4 relative for normal codes, 2^-10 * s below 2^-6 * s)
    D, P = 128, 64
    g = np.random.default_rng(7)
    n = 200
    x = (g.normal(0, 1, (n, D)) * g.uniform(0.01, 100, (n, 1))).astype(np.float32)
    k = _bf16(x)
    kf = (k.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    pool, stride = _pool((n + P - 1) // P, D, P, fp8=True)
    assert oracle.kcache_store(k, np.arange(n, dtype=np.int32), pool, stride,
                               (n + P - 1) // P, oracle.KV_E4M3, D=D, P=P) == 0
    for i in range(n):
        page, slot = divmod(i, P)
        c = pool[page * stride + slot * D: page * stride + slot * D + D]
        s = float(pool[page * stride + P * D + slot * 4: page * stride + P * D + slot * 4 + 4]
                  .view(np.float32)[0])
        deq = np.array([oracle.e4m3_to_double(int(v)) for v in c]) * s
        err = np.abs(deq - kf[i])
        bound = np.maximum(np.abs(kf[i]) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)
        assert (err <= bound).all(), i
        assert np.abs(kf[i]).max() / s == pytest.approx(448.0, rel=1e-6)
