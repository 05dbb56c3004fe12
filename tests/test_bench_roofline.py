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


def test_eta_line_reports_the_hbm_bound_with_the_fp32_fma_figure_beside_it():
    """The eta readout is set against the same bound as every line (HBM bytes
    versus bf16 tensor-peak flops, the slower); its fp32 CUDA-core figure is an
    extra field."""
    w = configs.PREFILL_1P3B
    r = bench.roofline(_Runner(w), 2.0, PEAKS, "measured", None, fp32_fma=True)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - r["algorithmic_bytes"] / 2.0e-3 / 1e9 / 6791.0) < 1e-4
    f = r["fp32_fma"]
    assert abs(f["peak"] - 152 * 128 * 2 * 2.07e9 / 1e12) < 0.1
    # 12 M (R + d) flops per position and head
    assert f["algorithmic_flops"] == 12.0 * 64 * 256 * 4 * 16 * 4096
    assert abs(f["frac"] - f["algorithmic_flops"] / 2.0e-3 / 1e12 / bench.FP32_TFLOPS_NOMINAL) < 1e-4


def test_bound_is_the_slower_of_bytes_and_flops():
    w = configs.PREFILL_1P3B
    r = bench.roofline(_Runner(w), 1.0, {"hbm_gbs": 1e6, "bf16_tflops": 1.0}, "measured", None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["bound_ms"] == round(1e3 * r["algorithmic_flops"] / 1e12, 5)


def test_every_workload_is_on_the_line():
    """The headline (1.3B-like prefill) plus the secondary lines cover all five
    workloads and the eta readout."""
    keys = {bench.line_key(w, f) for w, f in bench.SECONDARY}
    keys.add(bench.line_key(configs.PREFILL_1P3B, 0))
    assert keys == {"tiny_f32", "prefill_125m_bf16", "prefill_1p3b_bf16", "prefill_1p3b_bf16_eta",
                    "prefill_14k_bf16", "decode_bf16"}


def test_traffic_record_is_current_for_the_profiled_sources(tmp_path, monkeypatch):
    """A traffic record counts only while the kernels' sources hash to the profiled
    version; it carries the step's total over all of its launches."""
    import json
    sha = bench.sources_sha(bench.PREFILL_SOURCES)
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"prefill_1p3b_bf16": {"source_sha": sha, "step_bytes": 300,
                                 "kernels": {"a": 100, "b": 200}},
           "prefill_125m_bf16": {"source_sha": "stale", "step_bytes": 5, "kernels": {}}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    (tmp_path / "linear_token_mixer_sc_gb300").symlink_to(
        os.path.join(ROOT, "linear_token_mixer_sc_gb300"))
    assert bench.traffic_record("prefill_1p3b_bf16", bench.PREFILL_SOURCES) == (300, {"a": 100, "b": 200})
    assert bench.traffic_record("prefill_125m_bf16", bench.PREFILL_SOURCES) == (None, None)
    assert bench.traffic_record("decode_bf16", bench.DECODE_SOURCES) == (None, None)


def test_decode_bytes_count_the_state_twice():
    w = configs.DECODE
    S = bench.state_floats(w)
    assert S == 2 * 64 * 256 + 2 * 64 + 2 * 3 * 128
    assert bench.decode_bytes(w) == 256 * 16 * (2 * S * 4 + (3 * 128 + 128) * 2)
