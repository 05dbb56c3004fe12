"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source, builds it on
the CPU, and runs the pins against the mutant: at least one pin must fail.
Nothing here touches the real oracle library or the CUDA path.
"""
import importlib.util
import subprocess
from pathlib import Path

import pytest

from tests import test_oracle_pins as pins

ROOT = Path(__file__).resolve().parents[1]
SRC = ROOT / "oracle" / "ida_oracle.c"

# (name, text in ida_oracle.c, replacement)
MUTATIONS = [
    ("conjugated lambda", "row[c] = lam[m] * row[c] + Bv[m] * kr[c];",
     "row[c] = conj(lam[m]) * row[c] + Bv[m] * kr[c];"),
    ("value input without B", "row[R + j] = lam[m] * row[R + j] + Bv[m] * vr[j];",
     "row[R + j] = lam[m] * row[R + j] + vr[j];"),
    ("imaginary part read out", "double o = creal(acc);\n            out[(size_t)t * d + j]",
     "double o = cimag(acc);\n            out[(size_t)t * d + j]"),
    ("conv taps reversed", "acc += w[(size_t)c * W + j] * xv;", "acc += w[(size_t)c * W + (W - 1 - j)] * xv;"),
    ("unsquared norm", "xi[(size_t)t * C + c] = orc_silu(row[c]) / (sq + EPS_FEAT);",
     "xi[(size_t)t * C + c] = orc_silu(row[c]) / (sqrt(sq) + EPS_FEAT);"),
    ("RMS over the sum, not the mean", "        ms /= C;\n", "\n"),
    ("eta driven without B", "eta[m] = lam[m] * eta[m] + Bv[m];", "eta[m] = lam[m] * eta[m] + 1.0;"),
    ("query RMS-normed like the key", "    fmap(s, N, R, xq);\n",
     "    fmap(s, N, R, xq);\n    orc_rmsnorm_affine(xq, N, R, norm_w, bias, xq);\n"),
    ("l_2 map with the squared norm", "/ (sqrt(sq) + EPS_FEAT);", "/ (sq + EPS_FEAT);"),
    ("l_2 flag ignored", "flags & ORC_FEAT_L2, xq, kt, vt);", "0, xq, kt, vt);"),
    ("starting tails ignored", "flags, st, tin_q, tin_k, o, dn);", "flags, st, NULL, NULL, o, dn);"),
    ("final tails not reaching into the starting tails", "} else if (sin) {", "} else if (0) {"),
    ("starting eta ignored", "memcpy(st, sin, (size_t)2 * M * (RD + 1) * sizeof(double));",
     "memcpy(st, sin, (size_t)2 * M * RD * sizeof(double));"),
]

PIN_TESTS = [
    pins.test_conv_is_numpy_causal_convolution,
    pins.test_feature_map_squared_norm_invariants,
    pins.test_rmsnorm_unit_mean_square_and_affine,
    pins.test_prologue_golden_worked_example,
    pins.test_unit_feature_wiring,
    pins.test_recurrence_equals_bruteforce_double_sum,
    pins.test_lambda_one_single_mode_is_cumulative_sums,
    pins.test_lambda_zero_is_memoryless,
    pins.test_eta_readout_returns_constant_values,
    pins.test_prefill_from_state_one_position_is_decode_step,
    pins.test_feature_map_l2_invariants,
    pins.test_feature_map_l2_flag_reaches_both_feature_maps,
]


def _mutant(tmp_path, old, new):
    src = SRC.read_text()
    assert src.count(old) == 1, old
    mdir = tmp_path / "oracle_mutant"
    mdir.mkdir()
    (mdir / "ida_oracle.c").write_text(src.replace(old, new))
    so = mdir / "liboracle_ida.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-w",
                    str(mdir / "ida_oracle.c"), "-o", str(so), "-lm"], check=True)
    spec = importlib.util.spec_from_file_location("oracle_mutant_mod", ROOT / "oracle" / "ida_oracle.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC, mod._LIB_PATH, mod._lib = mdir / "ida_oracle.c", so, None
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new):
    mod = _mutant(tmp_path, old, new)
    monkeypatch.setattr(pins, "orc", mod)
    failed = []
    for t in PIN_TESTS:
        try:
            t()
        except AssertionError:
            failed.append(t.__name__)
    assert failed, f"no pin caught the planted mistake: {name}"
