"""The five synthetic workloads the mixer is checked and measured on.

Shapes stand in for the model sizes and context lengths of "Interdomain
Attention: Beyond Token-Level Key-Value Memory" (125M and 1.3B models, 4K
training context, 14K length extrapolation); the values are synthetic (see
``inputs``).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int          # prefill length (for decode: the seeding prefill)
    d: int
    R: int
    M: int
    W: int
    dtype: str      # "f32" or "bf16"
    seed: int
    eta: bool = False           # also run the eta-normalised readout
    final_state: bool = False   # prefill returns the final state
    decode_steps: int = 0       # > 0: recurrent decode workload

    @property
    def token_heads(self) -> int:
        return self.B * self.N * self.H


TINY_F32 = Workload("tiny_f32", B=1, H=2, N=256, d=32, R=32, M=16, W=4, dtype="f32", seed=1)
PREFILL_125M = Workload("prefill_125m_bf16", B=8, H=12, N=2048, d=64, R=64, M=64, W=4,
                        dtype="bf16", seed=2)
PREFILL_1P3B = Workload("prefill_1p3b_bf16", B=4, H=16, N=4096, d=128, R=128, M=64, W=4,
                        dtype="bf16", seed=3, eta=True)
PREFILL_14K = Workload("prefill_14k_bf16", B=1, H=16, N=14336, d=128, R=128, M=64, W=4,
                       dtype="bf16", seed=4, final_state=True)
DECODE = Workload("decode_bf16", B=256, H=16, N=4096, d=128, R=128, M=64, W=4,
                  dtype="bf16", seed=5, decode_steps=512)

ALL = {w.name: w for w in (TINY_F32, PREFILL_125M, PREFILL_1P3B, PREFILL_14K, DECODE)}
