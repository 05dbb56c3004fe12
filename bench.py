"""Throughput benchmark of the Interdomain Attention token mixer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one pass of the mixer over one batch of synthetic input: a
prefill (``ida_forward``) for the prefill workloads, one ``ida_decode_step``
over the whole batch for the decode workload.  The headline workload is the
largest single-GPU one, the 1.3B-like prefill at training context (B=4, H=16,
N=4096, R=d=128, M=64, bf16, denominator-free readout).  The same JSON line
carries, under ``workloads``, every other workload measured in the same run,
each with its own clocks and roofline: the tiny fp32 check, the 125M-like
prefill, the 1.3B-like prefill with the eta readout, the 14K-position prefill
returning its final state, and the recurrent decode step (batch 256, H=16,
state seeded by a 4096-position prefill).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream; between timed steps the L2 is flushed (a 512 MB
write and read-back outside the timed region), except where a step streams
more than four times the L2 (the decode state).  ``value`` is whole-job tokens/s
(a token is one position of one batch row, through all H heads).
``--impl reference`` times the CPU oracle instead (bounded sample per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from linear_token_mixer_sc_gb300 import configs, inputs  # noqa: E402

METRIC = "mixer tokens/s (prefill & decode) at 1 GB300; % of roofline (HBM/TC)"
L2_BYTES = 126 * 1024 * 1024
FLUSH_BYTES = 512 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal GB300 unit counts for the FP32 CUDA-core peak (the bound of the eta readout, which
# computes in fp32 on the CUDA cores): 152 SMs x 128 FP32 lanes x 2 flops (FMA) x 2.07 GHz
# maximum SM clock.
FP32_TFLOPS_NOMINAL = 152 * 128 * 2 * 2.07e9 / 1e12
PREFILL_SOURCES = ["ida_chunk.cu", "ida_seq.cu", "ida_common.cuh", "tc_sm103.cuh", "ida_api.cu"]
ETA_SOURCES = ["ida_seq_modes.cu", "ida_seq.cu", "ida_common.cuh", "ida_api.cu"]
DECODE_SOURCES = ["ida_decode.cu", "ida_common.cuh", "ida_api.cu"]
BACKWARD_SOURCES = ["ida_backward.cu", "ida_common.cuh", "ida_api.cu"]
IDEAL_SOURCES = ["ida_ideal.cu", "ida_common.cuh", "ida_api.cu"]
ROPE_SOURCES = ["ida_rope.cu", "ida_common.cuh", "ida_api.cu"]


# ---------------------------------------------------------------- helpers

def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def sources_sha(names) -> str:
    h = hashlib.sha256()
    for n in names:
        h.update((ROOT / "linear_token_mixer_sc_gb300" / "csrc" / n).read_bytes())
    return h.hexdigest()[:16]


def traffic_record(key: str, names):
    """DRAM bytes of one step (every launch of the step) from the committed ncu
    record, if the kernels' sources still hash to the profiled version; also the
    per-kernel figures it sums."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None, None
    rec = json.loads(p.read_text()).get(key)
    if not rec or rec.get("source_sha") != sources_sha(names):
        return None, None
    return rec.get("step_bytes"), rec.get("kernels")


def elem_bytes(dtype: str) -> int:
    return 4 if dtype == "f32" else 2


def prefill_bytes(w) -> int:
    """Compulsory HBM bytes of one prefill launch: read q, k, v once, write out once
    (plus the final state when it is returned)."""
    s = elem_bytes(w.dtype)
    b = w.B * w.H * w.N * ((2 * w.R + w.d) * s + w.d * s)
    if w.final_state:
        b += w.B * w.H * state_floats(w) * 4
    return b


def state_floats(w) -> int:
    n = 2 * w.M * (w.R + w.d) + 2 * w.M + 2 * (w.W - 1) * w.R
    return (n + 3) // 4 * 4


def decode_bytes(w) -> int:
    """One decode step: state read + write, q, k, v read, out written."""
    s = elem_bytes(w.dtype)
    return w.B * w.H * (2 * state_floats(w) * 4 + (2 * w.R + w.d) * s + w.d * s)


def resident_bytes(w) -> int:
    """Bytes a step touches that stay on the device between steps: the prefill's
    inputs and output, or the decode state."""
    if w.decode_steps:
        return w.B * w.H * state_floats(w) * 4
    s = elem_bytes(w.dtype)
    return w.B * w.H * w.N * (2 * w.R + 2 * w.d) * s


def flushes_l2(w) -> bool:
    """The L2 is flushed between timed steps unless a step streams more than four
    times the L2 (the decode state), where at most a quarter of it could be reused."""
    return resident_bytes(w) < 4 * L2_BYTES


def l2_note(w) -> str:
    return ("flushed between timed steps (512 MB write and read-back, outside the timed region)"
            if flushes_l2(w) else "inputs larger than L2 (the step streams more than 4x the L2)")


def mixer_flops(w, positions: int) -> float:
    """Algorithmic flops of the recurrent form: 12 M (R+d) per position and head
    (a 6-flop complex update of each state element, 2 flops per element for
    a = xi(q) U^T and 2 for Re(a Gamma))."""
    return 12.0 * w.M * (w.R + w.d) * positions


class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region: started (and its
    first sample awaited) before the warm-up, stopped after one more sample once the
    timed steps are done, so the samples bracket the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, device_index: int):
        self.proc = None
        self.idx = device_index
        self.lines = []
        self.thread = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def _wait_for(self, n, timeout_s):
        t0 = time.perf_counter()
        while len(self.lines) < n and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.005)

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        self._wait_for(1, 3.0)

    def stop(self):
        if self.proc is None:
            return None
        self._wait_for(len(self.lines) + 1, 1.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm

class Prefill:
    def __init__(self, w, dev, flags=0, from_state=False):
        from linear_token_mixer_sc_gb300 import binding
        self.b = binding
        self.w, self.dev, self.flags = w, dev, flags
        p = inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed)
        self.params_host = p
        self.pd = binding.params_to_device(p, dev)
        q, k, v = inputs.make_qkv(w.B, w.N, w.H, w.R, w.d, w.dtype, w.seed)
        self.host = [t.pin_memory() for t in (q, k, v)]
        self.q, self.k, self.v = (t.to(dev) for t in self.host)
        self.out = torch.empty((w.B, w.N, w.H, w.d), dtype=self.q.dtype, device=dev)
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.fs = (torch.empty((w.B, w.H, state_floats(w)), dtype=torch.float32, device=dev)
                   if w.final_state else None)
        # the workspace the library asks for (sequence segments on separate SMs); allocated once
        self.ws = binding.forward_workspace(self.q, self.v, self.pd, flags)
        self.in_bytes = sum(t.numel() * t.element_size() for t in self.host)
        # tensor-core path: readout kernels for the factorised- and the skewed-Gram heads, plus the
        # block state pass when split; the eta readout runs one sequential kernel
        if flags & binding.IDA_READOUT_ETA or w.dtype == "f32":
            self.launches_per_step = 1
        else:
            self.launches_per_step = 2 if self.ws is None else 3
        # continuing a sequence: the state after this same batch of positions (set-up, untimed)
        self.state_in = None
        if from_state:
            _, self.state_in = binding.ida_forward(self.q, self.k, self.v, self.pd, flags=flags,
                                                   final_state=True, workspace=self.ws)
            torch.cuda.synchronize(dev)
        # end to end: the host-memory entry point, its staging allocated once
        self.state_in_host = None if self.state_in is None else self.state_in.cpu().pin_memory()
        self.fs_host = None if self.fs is None else torch.empty(self.fs.shape, dtype=torch.float32).pin_memory()
        nst = binding.ida_forward_host_staging_bytes(w.B, w.H, w.N, w.d, w.R, w.M, binding._dtype_code(self.q),
                                                     w.W, flags)
        self.staging = torch.empty(max(nst, 16), dtype=torch.uint8, device=dev)

    def step(self):
        self.b.ida_forward(self.q, self.k, self.v, self.pd, out=self.out, final_state=self.fs,
                           flags=self.flags, workspace=self.ws, state_in=self.state_in)

    def step_e2e(self):
        # host buffers in, host buffers out: slices copied in, run and copied out on the
        # library's three streams (ida_forward_host)
        q, k, v = self.host
        self.b.ida_forward_host(q, k, v, self.pd, out=self.out_host, final_state=self.fs_host,
                                state_in=self.state_in_host, flags=self.flags, staging=self.staging)

    def e2e_bytes(self):
        bi = self.in_bytes + (0 if self.state_in_host is None else self.state_in_host.numel() * 4)
        bo = self.out.numel() * self.out.element_size() + (0 if self.fs_host is None else self.fs_host.numel() * 4)
        return bi, bo

    def tokens(self):
        return self.w.B * self.w.N

    def alg_bytes(self):
        extra = 0 if self.state_in is None else self.state_in.numel() * 4  # the start state, read once
        return prefill_bytes(self.w) + extra

    def flops(self):
        return mixer_flops(self.w, self.w.B * self.w.H * self.w.N)


class Decode:
    def __init__(self, w, dev, flags=0, seed_len=None):
        from linear_token_mixer_sc_gb300 import binding
        self.b = binding
        self.w, self.dev, self.flags = w, dev, flags
        p = inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed)
        self.pd = binding.params_to_device(p, dev)
        n0 = w.N if seed_len is None else seed_len
        q, k, v = inputs.make_qkv(w.B, n0, w.H, w.R, w.d, w.dtype, w.seed, device=dev)
        _, self.state = binding.ida_forward(q, k, v, self.pd, final_state=True)
        del q, k, v
        # a ring of pre-drawn tokens so that no generator runs inside the timed region
        self.ring = [inputs.make_tokens(w.B, w.H, w.R, w.d, w.dtype, w.seed, s, device=dev)
                     for s in range(8)]
        self.host_ring = [tuple(t.cpu().pin_memory() for t in r) for r in self.ring[:2]]
        self.dq, self.dk, self.dv = (torch.empty_like(t) for t in self.ring[0])
        self.out = torch.empty((w.B, w.H, w.d), dtype=self.ring[0][0].dtype, device=dev)
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.i = 0
        self.launches_per_step = 1
        torch.cuda.synchronize(dev)

    def step(self):
        q, k, v = self.ring[self.i % len(self.ring)]
        self.i += 1
        self.b.ida_decode_step(q, k, v, self.pd, self.state, out=self.out, flags=self.flags)

    def step_e2e(self):
        q, k, v = self.host_ring[self.i % 2]
        self.i += 1
        self.dq.copy_(q, non_blocking=True)
        self.dk.copy_(k, non_blocking=True)
        self.dv.copy_(v, non_blocking=True)
        self.b.ida_decode_step(self.dq, self.dk, self.dv, self.pd, self.state, out=self.out,
                               flags=self.flags)
        self.out_host.copy_(self.out, non_blocking=True)

    def e2e_bytes(self):
        r = self.host_ring[0]
        return sum(t.numel() * t.element_size() for t in r), self.out.numel() * self.out.element_size()

    def tokens(self):
        return self.w.B

    def alg_bytes(self):
        return decode_bytes(self.w)

    def flops(self):
        return mixer_flops(self.w, self.w.B * self.w.H)


class Backward:
    """One ida_backward call (the gradients of a prefill with respect to q, k, v and every
    parameter) over the workload's batch, from a seeded output gradient."""

    def __init__(self, w, dev, flags=0):
        from linear_token_mixer_sc_gb300 import binding
        self.b = binding
        self.w, self.dev, self.flags = w, dev, flags
        self.pd = binding.params_to_device(inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed), dev)
        q, k, v = inputs.make_qkv(w.B, w.N, w.H, w.R, w.d, w.dtype, w.seed)
        g = torch.Generator().manual_seed(w.seed + 1000)
        dout = torch.randn(w.B, w.N, w.H, w.d, generator=g).to(q.dtype)
        self.host = [t.pin_memory() for t in (q, k, v, dout)]
        self.q, self.k, self.v, self.dout = (t.to(dev) for t in self.host)
        nb = binding.ida_backward_workspace_bytes(w.B, w.H, w.N, w.d, w.R, w.M,
                                                  binding.IDA_BF16 if w.dtype == "bf16" else binding.IDA_F32,
                                                  w.W, flags)
        self.ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        self.grads = {"q": torch.empty_like(self.q), "k": torch.empty_like(self.k), "v": torch.empty_like(self.v)}
        self.grads.update({n: torch.empty_like(self.pd[n]) for n in ("conv_w", "norm_w", "bias", "lambda", "Bvec")})
        self.gq_host = torch.empty(self.q.shape, dtype=self.q.dtype).pin_memory()
        # features, forward scan, adjoint scan, position-local backward and parameter reduction,
        # plus the eta readout's scaling pass and the sum over mode slices when the modes
        # are split over CTAs (slices of 8 x floor(512 / (R + d rounded up to 32)) modes)
        slice_modes = 8 * (512 // ((w.R + w.d + 31) // 32 * 32))
        self.launches_per_step = 5 + (flags & 1) + (w.M > slice_modes)

    def step(self):
        self.b.ida_backward(self.q, self.k, self.v, self.pd, self.dout, flags=self.flags, workspace=self.ws,
                            grads=self.grads)

    def step_e2e(self):
        for src, dst in zip(self.host, (self.q, self.k, self.v, self.dout)):
            dst.copy_(src, non_blocking=True)
        self.step()
        self.gq_host.copy_(self.grads["q"], non_blocking=True)

    def e2e_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host), self.gq_host.numel() * self.gq_host.element_size()

    def tokens(self):
        return self.w.B * self.w.N

    def alg_bytes(self):
        """q, k, v and dout read once; dq, dk, dv written once."""
        s = elem_bytes(self.w.dtype)
        w = self.w
        return w.B * w.H * w.N * ((2 * w.R + 2 * w.d) * s + (2 * w.R + w.d) * s)

    def flops(self):
        """The forward recurrence recomputed plus its adjoint: three times the forward's
        12 M (R + d) per position and head."""
        return 3 * mixer_flops(self.w, self.w.B * self.w.H * self.w.N)


class Ideal:
    """One ida_forward_ideal call: the ideal interdomain layer on D random Fourier
    frequencies per head, at the 125M-like shape (R_in = d = 64, D = 32, so the feature
    width 2D equals R)."""

    D = 32

    def __init__(self, w, dev):
        from linear_token_mixer_sc_gb300 import binding
        self.b = binding
        self.w, self.dev = w, dev
        self.pd = binding.params_to_device(inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed), dev)
        q, k, v = inputs.make_qkv(w.B, w.N, w.H, w.R, w.d, w.dtype, w.seed)
        self.host = [t.pin_memory() for t in (q, k, v)]
        self.q, self.k, self.v = (t.to(dev) for t in self.host)
        self.omega = torch.from_numpy(inputs.make_omega(w.H, self.D, w.R, w.seed)).to(dev)
        self.out = torch.empty((w.B, w.N, w.H, w.d), dtype=self.q.dtype, device=dev)
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.launches_per_step = 1

    def step(self):
        self.b.ida_forward_ideal(self.q, self.k, self.v, self.omega, self.pd, out=self.out)

    def step_e2e(self):
        for src, dst in zip(self.host, (self.q, self.k, self.v)):
            dst.copy_(src, non_blocking=True)
        self.step()
        self.out_host.copy_(self.out, non_blocking=True)

    def e2e_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host), self.out.numel() * self.out.element_size()

    def tokens(self):
        return self.w.B * self.w.N

    def alg_bytes(self):
        return prefill_bytes(self.w)

    def flops(self):
        """The recurrent form on feature width 2D plus the Fourier features of q and k
        (D x R_in products each) per position and head."""
        w = self.w
        return (12.0 * w.M * (2 * self.D + w.d) + 4.0 * self.D * w.R) * w.B * w.H * w.N


class Rope:
    """One ida_rope call: rotary position embeddings on q and k of the prefill workload,
    in place (HBM-bound: q and k read and written once)."""

    def __init__(self, w, dev):
        from linear_token_mixer_sc_gb300 import binding
        self.b = binding
        self.w, self.dev = w, dev
        q, k, _ = inputs.make_qkv(w.B, w.N, w.H, w.R, w.d, w.dtype, w.seed)
        self.host = [t.pin_memory() for t in (q, k)]
        self.q, self.k = (t.to(dev) for t in self.host)
        self.back = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in self.host]
        self.launches_per_step = 1

    def step(self):
        self.b.ida_rope(self.q, self.k)

    def step_e2e(self):
        for src, dst in zip(self.host, (self.q, self.k)):
            dst.copy_(src, non_blocking=True)
        self.step()
        for src, dst in zip((self.q, self.k), self.back):
            dst.copy_(src, non_blocking=True)

    def e2e_bytes(self):
        n = sum(t.numel() * t.element_size() for t in self.host)
        return n, n

    def tokens(self):
        return self.w.B * self.w.N

    def alg_bytes(self):
        """q and k read once and written once."""
        return 2 * sum(t.numel() * t.element_size() for t in self.host)

    def flops(self):
        """Six flops per channel pair (four products, two sums), q and k."""
        w = self.w
        return 2 * 6.0 * (w.R // 2) * w.B * w.N * w.H


def time_steps(runner, steps, warmup, dev, flush, e2e=False, sampler=None):
    """Per-step CUDA-event times (ms) on the launching stream.  With ``flush`` the L2
    is flushed before every timed step, outside the timed region, by writing a 512 MB
    buffer and then reading it back: the write evicts the step's inputs, the read
    evicts the write's own dirty lines (their write-back happens there), so the timed
    step neither finds its inputs in L2 nor pays for another buffer's write-back."""
    stream = torch.cuda.current_stream(dev)
    fn = runner.step_e2e if e2e else runner.step
    scratch = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    sink = torch.empty((), dtype=torch.float32, device=dev)
    if sampler is not None:
        sampler.start()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        if scratch is not None:
            scratch.fill_(1.0)
            torch.sum(scratch, dim=0, out=sink)
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler is not None else None
    return [s.elapsed_time(e) for s, e in evs], clocks


def roofline(runner, ms_avg, peaks, peak_kind, traffic, fp32_fma=False):
    """The roofline record of one step: the slower of the algorithmic bytes at the
    measured HBM bandwidth and the algorithmic flops at the measured dense bf16
    tensor peak decides the bound; achieved = that quantity / the event-timed step.
    With ``fp32_fma`` (a path that computes on the CUDA cores in fp32 by design) the
    same flops are also set against the nominal fp32 FMA peak, as an extra field."""
    alg_b = runner.alg_bytes()
    fl = runner.flops()
    t_b = alg_b / (peaks["hbm_gbs"] * 1e9)
    t_f = fl / (peaks["bf16_tflops"] * 1e12)
    if t_b >= t_f:
        ach = alg_b / (ms_avg * 1e-3) / 1e9
        rec = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
               "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic,
               "algorithmic_bytes": alg_b, "peak_source": f"hbm_gbs ({peak_kind})"}
    else:
        ach = fl / (ms_avg * 1e-3) / 1e12
        rec = {"bound": "tensor", "achieved": round(ach, 2), "peak": peaks["bf16_tflops"],
               "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4), "traffic": traffic,
               "algorithmic_flops": fl, "peak_source": f"bf16_tflops ({peak_kind})"}
    rec["bound_ms"] = round(1e3 * max(t_b, t_f), 5)
    if fp32_fma:
        a32 = fl / (ms_avg * 1e-3) / 1e12
        rec["fp32_fma"] = {"achieved": round(a32, 2), "peak": round(FP32_TFLOPS_NOMINAL, 1),
                           "unit": "TFLOP/s", "frac": round(a32 / FP32_TFLOPS_NOMINAL, 4),
                           "algorithmic_flops": fl,
                           "peak_source": "fp32 FMA: 152 SMs x 128 lanes x 2 flops x 2.07 GHz (nominal)"}
    return rec


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(w, budget_s: float, cores: int, flags: int = 0):
    """Time the fp64 oracle on a bounded sample of the workload.

    Returns (tokens/s, description, seconds).  Prefill: the first k (b,h)
    units over all N positions; decode: k units for a few steps.
    """
    from oracle import ida_oracle as orc
    if w.decode_steps:
        B = min(w.B, max(1, cores))
        p = inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed)
        st = torch.zeros((B, w.H, orc.state_doubles(w.d, w.R, w.M, w.W)), dtype=torch.float64).numpy()
        n, t0 = 0, time.perf_counter()
        while True:
            q, k, v = inputs.make_tokens(B, w.H, w.R, w.d, w.dtype, w.seed, n)
            orc.decode_step(q, k, v, p, st, flags=flags, nthreads=cores)
            n += 1
            if time.perf_counter() - t0 > budget_s or n >= w.decode_steps:
                break
        dt = time.perf_counter() - t0
        return B * n / dt, f"{n} decode steps of batch {B} x {w.H} heads (of {w.B})", dt
    p = inputs.make_params(w.H, w.R, w.d, w.M, w.W, w.seed)
    # calibrate on one unit, then size the sample to the budget
    Bq = 1
    q, k, v = inputs.make_qkv(Bq, w.N, 1, w.R, w.d, w.dtype, w.seed)
    hp = {kk: vv[:, :1] if kk == "conv_w" else vv[:1] for kk, vv in p.items() if kk != "delta"}
    t0 = time.perf_counter()
    orc.forward(q, k, v, hp, flags=flags, nthreads=1)
    t1 = time.perf_counter() - t0
    units = max(1, min(w.B * w.H, int(budget_s * cores / max(t1, 1e-6))))
    Bs = max(1, min(w.B, math.ceil(units / w.H)))
    q, k, v = inputs.make_qkv(Bs, w.N, w.H, w.R, w.d, w.dtype, w.seed)
    ids = list(range(min(units, Bs * w.H)))
    t0 = time.perf_counter()
    orc.forward(q, k, v, p, flags=flags, units=ids, nthreads=cores)
    dt = time.perf_counter() - t0
    tok = len(ids) * w.N / w.H
    return tok / dt, f"{len(ids)} of {w.B * w.H} (b,h) units x {w.N} positions", dt


# ---------------------------------------------------------------- main

def dist_setup(n_gpus):
    """One process per GPU under torchrun: every rank runs the same per-GPU
    workload (weak scaling over independent (b,h) units); ranks exchange only
    their timings, never data."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        lr = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(lr)
        dist.init_process_group("nccl")
        return dist, dist.get_rank(), ws, lr
    return None, 0, 1, 0


def max_over_ranks(dist, x: float, dev) -> float:
    """The slowest rank's time (the job's time), on every rank."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world_size: int, tokens_per_rank: int, ms_max: float) -> float:
    """Whole-job tokens/s: all ranks' tokens over the slowest rank's step time."""
    return world_size * tokens_per_rank / (ms_max * 1e-3)


def line_key(w, flags=0, from_state=False) -> str:
    """Name of a measured line: the workload, with the readout and start noted."""
    return w.name + ("_eta" if flags & 1 else "") + ("_from_state" if from_state else "")


def sources_of(w, flags) -> list:
    if w.decode_steps:
        return DECODE_SOURCES
    if flags & 1 or w.dtype == "f32":
        return ETA_SOURCES
    return PREFILL_SOURCES


def measure(w, dev, steps, warmup, flags, dist, ws, peaks, peak_kind, e2e=True, seed_len=None,
            from_state=False, backward=False, ideal=False, rope=False):
    if rope:
        runner = Rope(w, dev)
    elif ideal:
        runner = Ideal(w, dev)
    elif backward:
        runner = Backward(w, dev, flags)
    elif w.decode_steps:
        runner = Decode(w, dev, flags, seed_len)
    else:
        runner = Prefill(w, dev, flags, from_state)
    flush = flushes_l2(w)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    wall0 = time.perf_counter()
    times, clocks = time_steps(runner, steps, warmup, dev, flush, sampler=sampler)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    ms = sum(times) / len(times)
    ms_all = max_over_ranks(dist, ms, dev)
    value = job_value(ws, runner.tokens(), ms_all)
    key = line_key(w, flags, from_state) + ("_backward" if backward else "") + ("_ideal" if ideal else "") + \
        ("_rope" if rope else "")
    traffic, per_kernel = traffic_record(key, BACKWARD_SOURCES if backward else IDEAL_SOURCES if ideal else
                                         ROPE_SOURCES if rope else sources_of(w, flags))
    rl = roofline(runner, ms, peaks, peak_kind, traffic,
                  fp32_fma=not rope and (backward or ideal or bool(flags & 1 and not w.decode_steps)
                                         or w.dtype == "f32"))
    if per_kernel:
        rl["traffic_kernels"] = per_kernel
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "R": w.R, "d": w.d, "M": w.M, "W": w.W,
           "dtype": w.dtype, "readout": "eta" if flags & 1 else "denominator-free",
           "l2": l2_note(w)}
    if backward:
        cfg["pass"] = "backward (gradients of q, k, v and every parameter)"
    if ideal:
        cfg["layer"] = f"ideal: random Fourier features, D = {Ideal.D} frequencies, eta ratio readout"
        cfg["readout"] = "eta"
    if rope:
        cfg = {"workload": w.name, "B": w.B, "N": w.N, "H": w.H, "R": w.R, "dtype": w.dtype,
               "op": "rotary position embeddings on q and k, in place (base 10000, positions 0..N-1)",
               "l2": l2_note(w)}
    elif w.decode_steps:
        cfg["seed_prefill_N"] = w.N if seed_len is None else seed_len
        del cfg["N"]
    else:
        cfg["start"] = "from a given state" if from_state else "zero state"
        cfg["final_state"] = bool(w.final_state)
    res = {"value": value, "unit": "tokens/s", "ms_per_step": ms_all, "steps": steps,
           "tokens_per_step": runner.tokens(), "wall_s": wall, "roofline": rl,
           "gpu_launches": runner.launches_per_step * steps, "clocks": clocks, "config": cfg}
    if e2e:
        et, _ = time_steps(runner, max(3, steps // 2), 2, dev, False, e2e=True)
        ems = max_over_ranks(dist, sum(et) / len(et), dev)
        bi, bo = runner.e2e_bytes()
        res["e2e"] = {"value": job_value(ws, runner.tokens(), ems), "unit": "tokens/s",
                      "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                      "ms_per_step": ems}
    del runner
    torch.cuda.empty_cache()
    return res


# The other workloads measured beside the headline one, in the same JSON line:
# (workload, flags).  Flag 1 is the eta readout.
SECONDARY = [(configs.TINY_F32, 0), (configs.PREFILL_125M, 0), (configs.PREFILL_1P3B, 1),
             (configs.PREFILL_14K, 0), (configs.DECODE, 0)]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=configs.PREFILL_1P3B.name, choices=sorted(configs.ALL))
    ap.add_argument("--eta", action="store_true", help="eta-normalised readout")
    ap.add_argument("--from-state", action="store_true",
                    help="prefill continuing from a given state (ida_forward_from)")
    ap.add_argument("--only", "--no-decode", dest="only", action="store_true",
                    help="measure the selected workload alone (no secondary lines)")
    ap.add_argument("--line", choices=["mixer", "backward", "ideal", "rope"], default="mixer",
                    help="what the main line measures on --workload: the mixer (default), its backward "
                         "pass, the ideal layer on Fourier features, or RoPE on q and k (for profiling "
                         "one of the secondary lines alone; no CPU leg)")
    ap.add_argument("--seed-len", type=int, default=None,
                    help="decode workload: length of the seeding prefill (default: the workload's 4096)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle CPU work for cpu_baseline (0: skip the CPU leg)")
    args = ap.parse_args()
    w = configs.ALL[args.workload]
    flags = 1 if args.eta else 0
    from_state = args.from_state and not w.decode_steps

    dist, rank, ws, lr = dist_setup(args.gpus)
    cores = os.cpu_count() or 1
    config = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "R": w.R, "d": w.d, "M": w.M,
              "W": w.W, "readout": "eta" if args.eta else "denominator-free",
              "parallelism": f"replicas x{ws} (independent (b,h) units, no collective)"}
    if not w.decode_steps:
        config["start"] = "from a given state" if from_state else "zero state"

    if args.impl == "reference":
        if rank != 0:
            return
        vals, desc, spent = [], "", 0.0
        budget = max(2.0, min(args.cpu_budget, 120.0 / max(1, args.steps + args.warmup)))
        for i in range(args.warmup + args.steps):
            v, desc, dt = oracle_sample(w, budget, cores, flags)
            if i >= args.warmup:
                vals.append(v)
                spent += dt
        value = sum(vals) / len(vals)
        config["l2"] = l2_note(w)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * spent / max(1, len(vals)), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                                 "kind": "oracle", "sample": desc,
                                 "host": f"{platform.machine()} x{cores}"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    dev = torch.device("cuda", lr)
    torch.cuda.set_device(dev)
    from linear_token_mixer_sc_gb300 import binding, build
    if rank == 0 or dist is None:
        build.build()
    if dist is not None:
        dist.barrier()
    binding.load()
    peaks, peak_kind = load_peaks()

    main_res = measure(w, dev, args.steps, args.warmup, flags, dist, ws, peaks, peak_kind,
                       seed_len=args.seed_len, from_state=from_state, backward=args.line == "backward",
                       ideal=args.line == "ideal", rope=args.line == "rope")
    others = {}
    if not args.only:
        for ow, of in SECONDARY:
            if (ow.name, of) == (w.name, flags) and not from_state:
                continue
            steps = max(args.steps, 64) if ow.decode_steps else args.steps
            r = measure(ow, dev, steps, args.warmup, of, dist, ws, peaks, peak_kind,
                        seed_len=args.seed_len)
            others[line_key(ow, of)] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps", "roofline",
                                                          "e2e", "gpu_launches", "clocks", "config")}
        # the backward pass of the 125M-like prefill (gradients for training the layer)
        bw = configs.PREFILL_125M
        r = measure(bw, dev, max(3, args.steps // 4), args.warmup, 0, dist, ws, peaks, peak_kind, backward=True)
        others[line_key(bw) + "_backward"] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps",
                                                                 "roofline", "e2e", "gpu_launches", "clocks",
                                                                 "config")}
        # the ideal layer on random Fourier features, at the same shape
        r = measure(bw, dev, args.steps, args.warmup, 0, dist, ws, peaks, peak_kind, ideal=True)
        others[line_key(bw) + "_ideal"] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps",
                                                              "roofline", "e2e", "gpu_launches", "clocks",
                                                              "config")}
        # rotary position embeddings on q and k of the 1.3B-like prefill
        rw = configs.PREFILL_1P3B
        r = measure(rw, dev, args.steps, args.warmup, 0, dist, ws, peaks, peak_kind, rope=True)
        others[line_key(rw) + "_rope"] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps",
                                                             "roofline", "e2e", "gpu_launches", "clocks",
                                                             "config")}
    if binding.ida_device_error() != 0:
        raise RuntimeError("a kernel reported a device error")

    if rank != 0:
        return
    cpu = None
    if args.cpu_budget > 0 and args.line == "mixer":
        cv, desc, _ = oracle_sample(w, args.cpu_budget, cores, flags)
        cpu = {"value": cv, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc,
               "host": f"{platform.machine()} x{cores}"}
    config["l2"] = l2_note(w)
    line = {"metric": METRIC, "value": main_res["value"], "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main_res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded; shapes of the pages' workloads)",
            "config": config, "roofline": main_res["roofline"], "cpu_baseline": cpu,
            "e2e": main_res["e2e"], "gpu_launches": main_res["gpu_launches"],
            "clocks": main_res["clocks"]}
    if args.line != "mixer":
        line["line"] = args.line
        line["config"] = main_res["config"]
    if others:
        line["workloads"] = others
    print(json.dumps(line))


if __name__ == "__main__":
    main()
