"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test ties the oracle to something it does not compute: hand-derived
values, a library routine in a special case where the definition reduces to
it, closed forms on the real page layout, invariants the definition implies,
and an exhaustive mask check.  Together they are chosen so that a dropped
term (ReLU, weight, scale), a wrong sign, a wrong page or slot index, or a
transposed operand fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from sparse_attention_paged_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_float(x):
    if x == "-inf":
        return -math.inf
    if x == "nan":
        return math.nan
    return float(x)


def run(oracle_mod, case, seqlens, kcache=None, block_table=None, **over):
    c = dict(case)
    c.update(over)
    out, status = oracle_mod.logits(
        c["q"], c["w"], c["kcache"] if kcache is None else kcache,
        c["kscale_offset"], c["page_stride"], c["num_pages"], c["kv_dtype"],
        c["block_table"] if block_table is None else block_table,
        c["bt_stride"], np.asarray(seqlens, dtype=np.int32), c["R"], c["H"],
        c["D"], c["P"], c["W"])
    return out, status


def golden_case(spec):
    H, D, P, W = spec["H"], spec["D"], spec["P"], spec["W"]
    q = bf16_bits(spec["q"]).reshape(-1, H, D)
    R = q.shape[0]
    w = np.asarray(spec["w"], dtype=np.float32).reshape(R, H)
    if spec["kv_dtype"] == "bf16":
        pages = spec["pages_bf16"]
        n = len(pages)
        pool = np.zeros((n, P * D), dtype=np.uint16)
        for k, v in pages.items():
            pool[int(k)] = bf16_bits(v).reshape(-1)
        kc = pool.view(np.uint8).reshape(-1)
        stride, koff, dt = P * D * 2, None, oracle_kv("bf16")
    else:
        pages = spec["pages_e4m3_codes"]
        n = len(pages)
        stride = P * D + 4 * P
        pool = np.zeros((n, stride), dtype=np.uint8)
        for k, v in pages.items():
            pool[int(k), : P * D] = np.asarray(v, dtype=np.uint8).reshape(-1)
            pool[int(k), P * D:] = np.asarray(spec["scales"][k], dtype=np.float32).view(np.uint8)
        kc = pool.reshape(-1)
        koff, dt = P * D, oracle_kv("e4m3")
    return dict(q=q, w=w, kcache=kc, kscale_offset=koff, page_stride=stride,
                num_pages=n, kv_dtype=dt,
                block_table=np.asarray(spec["block_table"], dtype=np.int32),
                bt_stride=W, R=R, H=H, D=D, P=P, W=W)


def oracle_kv(name):
    return 0 if name == "e4m3" else 1


# --------------------------------------------------------------------------
# 1. Hand-derived values

def test_hand_cases(oracle_mod):
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        spec = json.load(f)
    for c in spec["cases"]:
        case = golden_case(c)
        for run_ in c["runs"]:
            out, status = run(oracle_mod, case, run_["seqlens"])
            assert status == 0
            exp = np.array([[to_float(x) for x in row] for row in run_["expected"]])
            assert np.array_equal(out, exp), (c["name"], run_["seqlens"], out, exp)


def test_error_rows(oracle_mod):
    """Reading of a case the pages leave open: a length past the table is
    an error row of NaN; a page id outside the pool poisons its positions."""
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        c = json.load(f)["cases"][0]
    case = golden_case(c)
    out, status = run(oracle_mod, case, [5])
    assert status == oracle_mod.BAD_SEQLEN and np.isnan(out).all()
    bad = np.array([[1, 7]], dtype=np.int32)
    out, status = run(oracle_mod, case, [4], block_table=bad)
    assert status == oracle_mod.BAD_PAGE
    assert out[0, 0] == 0.5 and out[0, 1] == 0.0
    assert np.isnan(out[0, 2:]).all()
    # the bad entry is not needed when L stops before it
    out, status = run(oracle_mod, case, [2], block_table=bad)
    assert status == 0 and out[0, 0] == 0.5 and np.isneginf(out[0, 2:]).all()


# --------------------------------------------------------------------------
# 2. Bit decoders against library conversions

def test_e4m3_decoder_all_codes(oracle_mod):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle_mod.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2                                # 0x7F and 0xFF
    assert np.array_equal(mine[~nan], ref[~nan])
    assert oracle_mod.e4m3_to_double(0x7E) == 448.0
    assert oracle_mod.e4m3_to_double(0x01) == 2.0 ** -9


def test_bf16_decoder_all_patterns(oracle_mod):
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    mine = np.array([oracle_mod.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# --------------------------------------------------------------------------
# 3. Special cases that reduce to a library routine (numpy matmul)

def _identity_case(rng, kv, R=2, H=3, D=16, P=4, W=3):
    num_pages = R * W
    q = bf16_bits(rng.standard_normal((R, H, D)))
    w = rng.standard_normal((R, H)).astype(np.float32)
    bt = np.arange(num_pages, dtype=np.int32).reshape(R, W)
    if kv == 1:
        keys = bf16_bits(rng.standard_normal((num_pages, P, D)))
        kc = keys.view(np.uint8).reshape(-1)
        stride, koff = P * D * 2, None
        kdec = torch.from_numpy(keys.view(np.int16)).view(torch.bfloat16).double().numpy()
        scale = np.ones((num_pages, P))
    else:
        x = torch.from_numpy(rng.standard_normal((num_pages, P, D)).astype(np.float32))
        codes = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        scale = rng.uniform(0.5, 2.0, (num_pages, P)).astype(np.float32)
        stride = P * D + 4 * P
        pool = np.zeros((num_pages, stride), dtype=np.uint8)
        pool[:, : P * D] = codes.reshape(num_pages, -1)
        pool[:, P * D:] = scale.view(np.uint8).reshape(num_pages, -1)
        kc, koff = pool.reshape(-1), P * D
        kdec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
        scale = scale.astype(np.float64)
    case = dict(q=q, w=w, kcache=kc, kscale_offset=koff, page_stride=stride,
                num_pages=num_pages, kv_dtype=kv, block_table=bt, bt_stride=W,
                R=R, H=H, D=D, P=P, W=W)
    qdec = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).double().numpy()
    return case, qdec, kdec, scale


@pytest.mark.parametrize("kv", [0, 1])
def test_single_head_unit_weight_is_relu_matmul(oracle_mod, kv):
    """H=1, w=1: row r's logits are scale * relu(K_r @ q_r) with K_r the
    row's pages in table order -- a plain matrix-vector product."""
    rng = np.random.default_rng(1)
    case, qdec, kdec, scale = _identity_case(rng, kv, H=1)
    case["w"] = np.ones((case["R"], 1), dtype=np.float32)
    L = case["W"] * case["P"]
    out, st = run(oracle_mod, case, [L] * case["R"])
    assert st == 0
    for r in range(case["R"]):
        pages = case["block_table"][r]
        K = kdec[pages].reshape(-1, case["D"])           # [W*P, D]
        s = scale[pages].reshape(-1)
        ref = s * np.maximum(np.matmul(K, qdec[r, 0]), 0.0)
        np.testing.assert_allclose(out[r], ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("kv", [0, 1])
def test_one_hot_weights_select_a_head(oracle_mod, kv):
    """w = e_h picks head h alone: scale * relu(K @ q_h); any transposition
    of q (heads vs dims) or of the page (slots vs dims) breaks it."""
    rng = np.random.default_rng(2)
    case, qdec, kdec, scale = _identity_case(rng, kv, H=3, D=16)
    L = case["W"] * case["P"]
    for h in range(case["H"]):
        w = np.zeros((case["R"], case["H"]), dtype=np.float32)
        w[:, h] = 1.0
        out, st = run(oracle_mod, case, [L] * case["R"], w=w)
        assert st == 0
        for r in range(case["R"]):
            pages = case["block_table"][r]
            K = kdec[pages].reshape(-1, case["D"])
            ref = scale[pages].reshape(-1) * np.maximum(K @ qdec[r, h], 0.0)
            np.testing.assert_allclose(out[r], ref, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# 4. Closed forms on the real page layout (H=64, D=128, P=64)

def test_closed_form_fp8_fused_block(oracle_mod):
    """All keys 1.0 (e4m3 0x38), q = 2^-7 everywhere, w = 2^-6 for every
    head: each dot is 128 * 2^-7 = 1, the head sum is 64 * 2^-6 = 1, so the
    logit equals the position's scale, read from byte offset 8,192 of its
    8,448-byte page."""
    H, D, P, W, R = 64, 128, 64, 3, 2
    num_pages = 5
    pool = np.zeros((num_pages, wl.FP8_PAGE_BYTES), dtype=np.uint8)
    pool[:, : P * D] = 0x38
    scales = (100.0 * np.arange(num_pages)[:, None] + np.arange(P)[None, :] + 1).astype(np.float32)
    pool[:, wl.FP8_SCALE_OFFSET:] = scales.view(np.uint8)
    q = np.full((R, H, D), 0x3C00, dtype=np.uint16)          # bf16 2^-7
    w = np.full((R, H), 2.0 ** -6, dtype=np.float32)
    bt = np.array([[4, 0, 2], [1, 3, 4]], dtype=np.int32)
    seqlens = np.array([150, 192], dtype=np.int32)
    out, st = oracle_mod.logits(q, w, pool.reshape(-1), wl.FP8_SCALE_OFFSET,
                                wl.FP8_PAGE_BYTES, num_pages, 0, bt, W, seqlens,
                                R, H, D, P, W)
    assert st == 0
    for r in range(R):
        exp = scales[bt[r]].reshape(-1).astype(np.float64)
        exp[seqlens[r]:] = -np.inf
        assert np.array_equal(out[r], exp)


def test_closed_form_bf16_alternating_sign(oracle_mod):
    """bf16 keys k[d] = (-1)^d * c_t, q[h, d] = 1: every dot is 0 (relu 0).
    Flip to q[h, d] = (-1)^d: every dot is 128 * c_t; with c_t = 2^-7 * (t+1)
    ... the logit is (t+1) * sum_h w_h.  A dropped ReLU, a wrong slot index or
    a reversed d index changes the result."""
    H, D, P, W = 64, 128, 64, 2
    num_pages = 2
    T = W * P
    c = (np.arange(T) % 64 + 1).astype(np.float32) * 2.0 ** -7    # exact in bf16
    sign = np.where(np.arange(D) % 2 == 0, 1.0, -1.0).astype(np.float32)
    keys = bf16_bits(c[:, None] * sign[None, :]).reshape(num_pages, P, D)
    kc = keys.view(np.uint8).reshape(-1)
    w = np.linspace(-1, 2, H).astype(np.float32)[None, :]
    bt = np.array([[1, 0]], dtype=np.int32)
    ones = np.ones((1, H, D), dtype=np.float32)
    out0, st = oracle_mod.logits(bf16_bits(ones), w, kc, None, wl.BF16_PAGE_BYTES,
                                 num_pages, 1, bt, W, np.array([T], np.int32), 1, H, D, P, W)
    assert st == 0 and np.array_equal(out0[0], np.zeros(T))
    alt = np.broadcast_to(sign, (1, H, D))
    out1, st = oracle_mod.logits(bf16_bits(alt), w, kc, None, wl.BF16_PAGE_BYTES,
                                 num_pages, 1, bt, W, np.array([T], np.int32), 1, H, D, P, W)
    # position t reads physical page bt[t // P] slot t % P, whose c is (slot+1)/128
    slot = np.arange(T) % P
    exp = (slot + 1).astype(np.float64) * float(np.sum(w.astype(np.float64)))
    np.testing.assert_allclose(out1[0], exp, rtol=1e-14)


# --------------------------------------------------------------------------
# 5. Invariants of the definition

def _random_case(seed, kv=0, R=3, W=4, pool_extra=3):
    g = np.random.default_rng(seed)
    H, D, P = 64, 128, 64
    num_pages = R * W + pool_extra
    q = bf16_bits(g.standard_normal((R, H, D)))
    w = (g.standard_normal((R, H)) / 8).astype(np.float32)
    if kv == 0:
        stride = wl.FP8_PAGE_BYTES
        pool = np.zeros((num_pages, stride), dtype=np.uint8)
        x = torch.from_numpy(g.standard_normal((num_pages, P * D)).astype(np.float32))
        pool[:, : P * D] = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        pool[:, P * D:] = g.uniform(0.5, 2, (num_pages, P)).astype(np.float32).view(np.uint8)
        koff = wl.FP8_SCALE_OFFSET
    else:
        stride = wl.BF16_PAGE_BYTES
        pool = bf16_bits(g.standard_normal((num_pages, P * D))).view(np.uint8)
        koff = None
    bt = g.permutation(num_pages)[: R * W].astype(np.int32).reshape(R, W)
    seqlens = g.integers(1, W * P + 1, R).astype(np.int32)
    return dict(q=q, w=w, kcache=pool.reshape(-1), kscale_offset=koff,
                page_stride=stride, num_pages=num_pages, kv_dtype=kv,
                block_table=bt, bt_stride=W, R=R, H=H, D=D, P=P, W=W), seqlens


@pytest.mark.parametrize("kv", [0, 1])
def test_mask_is_exactly_positions_at_or_past_length(oracle_mod, kv):
    case, _ = _random_case(3, kv, R=1, W=3)
    T = case["W"] * case["P"]
    for L in [0, 1, 63, 64, 65, T - 1, T]:
        out, st = run(oracle_mod, case, [L])
        assert st == 0
        assert np.array_equal(np.isneginf(out[0]), np.arange(T) >= L), L
        assert np.isfinite(out[0, :L]).all()


@pytest.mark.parametrize("kv", [0, 1])
def test_page_permutation_invariance(oracle_mod, kv):
    """Moving physical pages and remapping the table leaves out bit-identical."""
    case, seqlens = _random_case(4, kv)
    out, st = run(oracle_mod, case, seqlens)
    g = np.random.default_rng(5)
    perm = g.permutation(case["num_pages"])           # new slot of old page p
    pool = case["kcache"].reshape(case["num_pages"], -1)
    moved = np.empty_like(pool)
    moved[perm] = pool
    bt2 = perm[case["block_table"]].astype(np.int32)
    out2, st2 = run(oracle_mod, case, seqlens, kcache=moved.reshape(-1), block_table=bt2)
    assert st == st2 == 0
    assert np.array_equal(out, out2)


def test_linearity_in_weights(oracle_mod):
    case, seqlens = _random_case(6, 0)
    out, _ = run(oracle_mod, case, seqlens)
    fin = np.isfinite(out)
    # powers of two (either sign) scale w exactly in fp32, so the result is
    # exactly alpha * out
    for alpha in [2.0, -0.5, -4.0]:
        o2, _ = run(oracle_mod, case, seqlens, w=(case["w"] * alpha).astype(np.float32))
        assert np.array_equal(o2[fin], alpha * out[fin])
        assert np.array_equal(np.isneginf(o2), ~fin)
    # additivity: dyadic weights with few bits, so w1 + w2 is exact in fp32
    g = np.random.default_rng(7)
    w1 = (np.round(g.standard_normal(case["w"].shape) * 256) / 2048).astype(np.float32)
    w2 = (np.round(g.standard_normal(case["w"].shape) * 256) / 2048).astype(np.float32)
    assert np.array_equal(w1.astype(np.float64) + w2, (w1 + w2).astype(np.float64))
    oa, _ = run(oracle_mod, case, seqlens, w=w1)
    ob, _ = run(oracle_mod, case, seqlens, w=w2)
    oc, _ = run(oracle_mod, case, seqlens, w=(w1 + w2).astype(np.float32))
    np.testing.assert_allclose(oc[fin], (oa + ob)[fin], rtol=1e-12,
                               atol=1e-12 * np.abs(oc[fin]).max())


def test_positive_homogeneity_in_q(oracle_mod):
    case, seqlens = _random_case(8, 1)
    out, _ = run(oracle_mod, case, seqlens)
    fin = np.isfinite(out)
    q4 = bf16_bits(torch.from_numpy(case["q"].view(np.int16)).view(torch.bfloat16).float().numpy() * 4)
    o4, _ = run(oracle_mod, case, seqlens, q=q4)
    assert np.array_equal(o4[fin], 4 * out[fin])
    qn = bf16_bits(-torch.from_numpy(case["q"].view(np.int16)).view(torch.bfloat16).float().numpy())
    on, _ = run(oracle_mod, case, seqlens, q=qn)
    assert not np.allclose(on[fin], -out[fin])          # ReLU is not odd


def test_scale_doubling_doubles_that_position(oracle_mod):
    case, seqlens = _random_case(9, 0, R=1, W=2)
    seqlens = np.array([128], np.int32)
    out, _ = run(oracle_mod, case, seqlens)
    pool = case["kcache"].reshape(case["num_pages"], -1).copy()
    phys = case["block_table"][0, 1]
    sc = pool[phys, wl.FP8_SCALE_OFFSET:].view(np.float32)
    sc[5] *= 2
    o2, _ = run(oracle_mod, case, seqlens, kcache=pool.reshape(-1))
    t = 64 + 5
    assert o2[0, t] == 2 * out[0, t]
    other = np.arange(128) != t
    assert np.array_equal(o2[0, other], out[0, other])


def test_head_additivity(oracle_mod):
    case, seqlens = _random_case(10, 1, R=2, W=2)
    out, _ = run(oracle_mod, case, seqlens)
    fin = np.isfinite(out)
    total = np.zeros_like(out)
    for h in range(case["H"]):
        wh = np.zeros_like(case["w"])
        wh[:, h] = case["w"][:, h]
        oh, _ = run(oracle_mod, case, seqlens, w=wh)
        total += np.where(fin, oh, 0)
    np.testing.assert_allclose(out[fin], total[fin], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("kv", [0, 1])
def test_widening_table_with_poison_changes_nothing_valid(oracle_mod, kv):
    case, seqlens = _random_case(11, kv, R=2, W=3)
    out, _ = run(oracle_mod, case, seqlens)
    # add a NaN page and widen the table with entries that point at it
    pool = case["kcache"].reshape(case["num_pages"], -1)
    poison = np.full((1, pool.shape[1]), 0xFF, dtype=np.uint8)       # NaN bytes
    pool2 = np.concatenate([pool, poison]).reshape(-1)
    W2 = case["W"] + 5
    bt2 = np.full((case["R"], W2), case["num_pages"], dtype=np.int32)
    bt2[:, : case["W"]] = case["block_table"]
    o2, st = run(oracle_mod, case, seqlens, kcache=pool2, block_table=bt2,
                 W=W2, bt_stride=W2, num_pages=case["num_pages"] + 1)
    assert st == 0
    T = case["W"] * case["P"]
    assert np.array_equal(o2[:, :T], out)
    assert np.isneginf(o2[:, T:]).all()


def test_prefill_equals_decode_with_rows_repeated(oracle_mod):
    """Prefill (rows share one table row, bt_stride 0, causal lengths) is the
    decode definition with the table row repeated."""
    case, _ = _random_case(12, 1, R=4, W=3)
    T = case["W"] * case["P"]
    seqlens = np.array([T - 40, T - 39, T - 38, T - 37], dtype=np.int32)
    bt_shared = case["block_table"][:1]
    o_pre, st = run(oracle_mod, case, seqlens, block_table=bt_shared, bt_stride=0)
    rep = np.repeat(bt_shared, case["R"], axis=0)
    o_dec, st2 = run(oracle_mod, case, seqlens, block_table=rep)
    assert st == st2 == 0
    assert np.array_equal(o_pre, o_dec)


def test_threads_do_not_change_result(oracle_mod):
    case, seqlens = _random_case(13, 0, R=5, W=2)
    outs = []
    for nt in [1, 2, 5, 0]:
        o, _ = oracle_mod.logits(case["q"], case["w"], case["kcache"], case["kscale_offset"],
                                 case["page_stride"], case["num_pages"], 0,
                                 case["block_table"], case["W"], seqlens, case["R"],
                                 64, 128, 64, case["W"], nthreads=nt)
        outs.append(o)
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


# --------------------------------------------------------------------------
# 6. The generator's layouts feed the oracle as documented

def test_generator_layout_small_config(oracle_mod):
    """cfg1 through the oracle: finite below L, -inf at and past L, no NaN
    (a NaN would mean an unreferenced, poisoned page was read)."""
    w_ = wl.cfg1()
    out, st = oracle_mod.logits(w_.q_bits, w_.w, w_.kcache, w_.kscale_offset,
                                w_.page_stride, w_.num_pages, w_.kv_dtype,
                                w_.block_table, w_.bt_stride, w_.seqlens,
                                w_.R, 64, 128, 64, w_.W)
    assert st == 0
    L = int(w_.seqlens[0])
    assert np.isfinite(out[0, :L]).all() and np.isneginf(out[0, L:]).all()
    assert not np.isnan(out).any()
