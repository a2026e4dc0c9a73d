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
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), str(src), "-lm"], check=True)
    return oracle.load_library(str(so))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
def test_unmutated_copy_passes(tmp_path):
    with open(os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")) as f:
        text = f.read()
    assert _golden_passes(_compile(text, tmp_path, "clean"))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(tmp_path, name):
    with open(os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")) as f:
        text = f.read()
    old, new = MUTATIONS[name]
    assert text.count(old) == 1, f"mutation anchor not found: {old}"
    lib = _compile(text.replace(old, new), tmp_path, "mutant")
    assert not _golden_passes(lib), f"golden cases missed mutation: {name}"
