"""Host logic of bench.py's roofline record (no GPU): which bound a line reports,
and the algorithmic bytes and flops it divides by."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linear_token_mixer_sc_gb300 import configs  # noqa: E402

PEAKS = {"hbm_gbs": 6791.0, "bf16_tflops": 1900.0}


class _Runner:
    def __init__(self, w, state_bytes=0):
        self.w, self.state_bytes = w, state_bytes

    def alg_bytes(self):
        return bench.prefill_bytes(self.w) + self.state_bytes

    def flops(self):
        return bench.mixer_flops(self.w, self.w.B * self.w.H * self.w.N)


def test_prefill_is_hbm_bound_with_compulsory_bytes():
    w = configs.PREFILL_125M
    r = bench.roofline(_Runner(w), 0.2, PEAKS, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    # q, k, v read once and out written once, bf16: B N H ((2R + d) + d) * 2 bytes
    assert r["algorithmic_bytes"] == 8 * 2048 * 12 * (3 * 64 + 64) * 2
    assert abs(r["achieved"] - r["algorithmic_bytes"] / 0.2e-3 / 1e9) < 0.1
    assert abs(r["frac"] - r["achieved"] / 6791.0) < 1e-4


def test_eta_line_reports_the_fp32_fma_bound():
    w = configs.PREFILL_1P3B
    r = bench.roofline(_Runner(w), 2.0, PEAKS, "measured", None, kernel_bound="alu")
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert abs(r["peak"] - 152 * 128 * 2 * 2.07e9 / 1e12) < 0.1
    # 12 M (R + d) flops per position and head
    assert r["algorithmic_flops"] == 12.0 * 64 * 256 * 4 * 16 * 4096
    assert abs(r["frac"] - r["algorithmic_flops"] / 2.0e-3 / 1e12 / bench.FP32_TFLOPS_NOMINAL) < 1e-4


def test_decode_bytes_count_the_state_twice():
    w = configs.DECODE
    S = bench.state_floats(w)
    assert S == 2 * 64 * 256 + 2 * 64 + 2 * 3 * 128
    assert bench.decode_bytes(w) == 256 * 16 * (2 * S * 4 + (3 * 128 + 128) * 2)
