"""Plant plausible mistakes in a copy of the oracle and show the hand-derived
golden cases reject every one (CPU only).

Each mutation is a one-line change to a private copy of the C source; the
committed oracle is never modified.
"""
import json
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import GOLDEN, golden_case, to_float

MUTATIONS = {
    "relu dropped": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "head weight dropped": ("acc += (double)J->w[(long long)r * J->H + h] * relu;", "acc += relu;"),
    "scale dropped": ("o[t] = key_scale(J, phys, j) * acc;", "o[t] = acc;"),
    "block table ignored": ("int phys = bt[page];", "int phys = page;"),
    "mask off by one": ("if (t >= L) {", "if (t > L) {"),
    "e4m3 exponent bias": ("expo - 10)", "expo - 9)"),
    "e4m3 sign dropped": ("return sign ? -mag : mag;", "return mag;"),
    "e4m3 subnormal scale": ("mag = ldexp((double)man, -9);", "mag = ldexp((double)man, -10);"),
    "scale slot reversed": ("+ 4LL * j, sizeof s", "+ 4LL * (J->P - 1 - j), sizeof s"),
    "slot index shifted": ("int j = (int)(t % J->P);", "int j = (int)((t + 1) % J->P);"),
    "q dims reversed": ("dsa_oracle_bf16_to_double(qh[d])", "dsa_oracle_bf16_to_double(qh[J->D - 1 - d])"),
}


STORE_MUTATIONS = {
    "e4m3 ties away from even": ("(d == best_d && (c & 1) == 0 && (best & 1) == 1)", "(d == best_d)"),
    "e4m3 saturates to the NaN code": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);",
                                       "if (a >= 448.0) return (uint8_t)(sign | 0x7F);"),
    "e4m3 largest code unreachable": ("for (int c = 1; c <= 0x7E; ++c) {", "for (int c = 1; c < 0x7E; ++c) {"),
    "e4m3 zero loses its sign": ("const uint8_t sign = signbit(x) ? 0x80 : 0x00;", "const uint8_t sign = (x < 0.0f) ? 0x80 : 0x00;"),
    "store scale divisor": ("amax / 448.0f : 1.0f;", "amax / 240.0f : 1.0f;"),
    "store scale slot": ("memcpy(pg + (long long)P * D + (long long)slot * 4, &sv, 4);",
                         "memcpy(pg + (long long)P * D + (long long)(P - 1 - slot) * 4, &sv, 4);"),
    "store bad slot accepted": ("if (page >= num_pages) {", "if (page > num_pages) {"),
}


def _store_golden_passes(lib) -> bool:
    """The store pins of test_oracle_store_pins, run against `lib`."""
    from tests.test_oracle_store_pins import _bf16
    for c in range(256):
        if c & 0x7F != 0x7F and lib.dsa_oracle_e4m3_encode(lib.dsa_oracle_e4m3_to_double(c)) != c:
            return False
    vals = [lib.dsa_oracle_e4m3_to_double(c) for c in range(0x7F)]
    for c in range(0x7E):
        m = (vals[c] + vals[c + 1]) / 2
        if lib.dsa_oracle_e4m3_encode(m) != (c if c % 2 == 0 else c + 1):
            return False
    if lib.dsa_oracle_e4m3_encode(470.0) != 0x7E or lib.dsa_oracle_e4m3_encode(-2.0 ** -11) != 0x80:
        return False
    D, P = 4, 2
    stride = P * (D + 4)
    pool = np.full(3 * stride, 0xA5, dtype=np.uint8)
    k = np.stack([_bf16([448.0, 1.0, -3.0, 0.0]), _bf16([2.0, -0.5, 0.25, 1.75]),
                  _bf16([1.0, 1.0, 1.0, 1.0])])
    st = oracle.kcache_store(k, np.array([3, 0, 4], np.int32), pool, stride, 2, oracle.KV_E4M3,
                             D=D, P=P, lib=lib)
    if st != oracle.BAD_PAGE:
        return False
    if list(pool[stride + D: stride + 2 * D]) != [0x7E, 0x38, 0xC4, 0x00]:
        return False
    if list(pool[0:D]) != [0x7E, 0xEE, 0x66, 0x7C]:
        return False
    s0 = pool[P * D: P * D + 4].view(np.float32)[0]
    s1 = pool[stride + P * D + 4: stride + P * D + 8].view(np.float32)[0]
    return bool(s0 == np.float32(2.0) / np.float32(448.0) and s1 == np.float32(1.0)
                and (pool[2 * stride:] == 0xA5).all())


def _golden_passes(lib) -> bool:
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        spec = json.load(f)
    for c in spec["cases"]:
        case = golden_case(c)
        for run_ in c["runs"]:
            out, _ = oracle.logits(
                case["q"], case["w"], case["kcache"], case["kscale_offset"],
                case["page_stride"], case["num_pages"], case["kv_dtype"],
                case["block_table"], case["bt_stride"],
                np.asarray(run_["seqlens"], np.int32), case["R"], case["H"],
                case["D"], case["P"], case["W"], lib=lib)
            exp = np.array([[to_float(x) for x in row] for row in run_["expected"]])
            if not np.array_equal(out, exp):
                return False
    return True


def _compile(src_text: str, tmp_path, tag: str):
    src = tmp_path / f"{tag}.c"
    so = tmp_path / f"lib{tag}.so"
    src.write_text(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    "-o", str(so), str(src), "-lm"], check=True)
    return oracle.load_library(str(so))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
def test_unmutated_copy_passes(tmp_path):
    with open(os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")) as f:
        text = f.read()
    lib = _compile(text, tmp_path, "clean")
    assert _golden_passes(lib)
    assert _store_golden_passes(lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(tmp_path, name):
    with open(os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")) as f:
        text = f.read()
    old, new = MUTATIONS[name]
    assert text.count(old) == 1, f"mutation anchor not found: {old}"
    lib = _compile(text.replace(old, new), tmp_path, "mutant")
    assert not _golden_passes(lib), f"golden cases missed mutation: {name}"


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
@pytest.mark.parametrize("name", sorted(STORE_MUTATIONS))
def test_store_mutant_is_caught(tmp_path, name):
    with open(os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")) as f:
        text = f.read()
    old, new = STORE_MUTATIONS[name]
    assert text.count(old) == 1, f"mutation anchor not found: {old}"
    lib = _compile(text.replace(old, new), tmp_path, "mutant")
    assert not _store_golden_passes(lib), f"store pins missed mutation: {name}"
