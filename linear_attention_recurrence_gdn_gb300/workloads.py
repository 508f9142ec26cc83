"""Seeded synthetic inputs for the GDN recurrence.

This module only draws random numbers; it holds none of the method's arithmetic.  The same
tensors feed the CUDA library and the fp64 oracle, so both sides see identical bits.

Recipe (per workload): a CPU ``torch.Generator`` seeded with ``seed``; draws in the fixed
order q, k, v, z, log_decay, beta, s0, GN; activations are drawn in float32 and then cast to
the workload's activation dtype; gates, s0 and GN stay float32.

* q, k, v, z ~ N(0, 1)                         (standard deviation 1)
* log_decay = -exp(U(lo, hi))                  so alpha = exp(log_decay) lies in (0, 1)
* beta = sigmoid(N(0, 1))                      in (0, 1)
* s0 ~ N(0, s0_std) or absent (zeros)          f32 [B, Hv, Dv, Dk]
* GN = 1 + N(0, 0.1)                           f32 [Dv]

The shapes follow the Qwen-style GDN layer geometry (GDNShape: num_key_heads,
num_value_heads, key_head_dim, value_head_dim).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    act: str                      # "f32" | "bf16" | "f16"  (q, k, v, z)
    head_major: bool
    log_decay_range: tuple        # (lo, hi): log_decay = -exp(U(lo, hi))
    s0_std: float | None          # None: no initial state (zeros)
    api: str                      # "decode" | "scan"
    seed: int

    @property
    def act_dtype(self) -> torch.dtype:
        return _DTYPES[self.act]

    @property
    def elem_bytes(self) -> int:
        return {"f32": 4, "bf16": 2, "f16": 2}[self.act]

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def as_config(self) -> dict:
        return {"workload": self.name, "B": self.B, "S": self.S, "Hk": self.Hk, "Hv": self.Hv,
                "Dk": self.Dk, "Dv": self.Dv, "act_dtype": self.act,
                "head_major": self.head_major}


# The five workloads: one tiny case the oracle finishes instantly, two decode steps and two
# prefill scans at Qwen-style layer sizes.
TINY = Workload("tiny_f32_b1_s8_h2_d16", B=1, S=8, Hk=2, Hv=2, Dk=16, Dv=16, act="f32",
                head_major=False, log_decay_range=(-3.0, 0.0), s0_std=0.1, api="scan",
                seed=1001)
DECODE_B64 = Workload("decode_bf16_b64_hk16_hv32_d128", B=64, S=1, Hk=16, Hv=32, Dk=128,
                      Dv=128, act="bf16", head_major=False, log_decay_range=(-4.0, 0.0),
                      s0_std=0.02, api="decode", seed=1002)
DECODE_B256_HM = Workload("decode_bf16_b256_hk16_hv32_d128_head_major", B=256, S=1, Hk=16,
                          Hv=32, Dk=128, Dv=128, act="bf16", head_major=True,
                          log_decay_range=(-4.0, 0.0), s0_std=0.02, api="decode", seed=1003)
PREFILL_B4 = Workload("prefill_bf16_b4_s4096_hk16_hv32_d128", B=4, S=4096, Hk=16, Hv=32,
                      Dk=128, Dv=128, act="bf16", head_major=False,
                      log_decay_range=(-4.0, 0.0), s0_std=None, api="scan", seed=1004)
LONG_B2 = Workload("long_f16_b2_s16384_hk8_hv32_d128", B=2, S=16384, Hk=8, Hv=32, Dk=128,
                   Dv=128, act="f16", head_major=False, log_decay_range=(-8.0, -3.0),
                   s0_std=0.02, api="scan", seed=1005)

WORKLOADS = [TINY, DECODE_B64, DECODE_B256_HM, PREFILL_B4, LONG_B2]
BY_NAME = {w.name: w for w in WORKLOADS}


def shapes(w: Workload) -> dict:
    """Tensor shapes of every operand of ``w`` (layout chosen by ``head_major``)."""
    if w.head_major:
        qk = (w.B, w.Hk, w.S, w.Dk)
        vz = (w.B, w.Hv, w.S, w.Dv)
        gate = (w.B, w.Hv, w.S)
    else:
        qk = (w.B, w.S, w.Hk, w.Dk)
        vz = (w.B, w.S, w.Hv, w.Dv)
        gate = (w.B, w.S, w.Hv)
    return {"q": qk, "k": qk, "v": vz, "z": vz, "y": vz, "log_decay": gate, "beta": gate,
            "state": (w.B, w.Hv, w.Dv, w.Dk), "gn": (w.Dv,)}


def make_inputs(w: Workload, *, seed: int | None = None,
                gate_dtype: torch.dtype = torch.float32) -> dict:
    """Draw the inputs of ``w`` on the CPU.  Returns a dict of tensors.

    Keys: q, k, v, z, log_decay, beta, s0 (None when ``s0_std`` is None), gn.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed if seed is None else seed)
    sh = shapes(w)

    def normal(shape, std=1.0):
        return torch.randn(shape, generator=gen, dtype=torch.float32) * std

    q = normal(sh["q"]).to(w.act_dtype)
    k = normal(sh["k"]).to(w.act_dtype)
    v = normal(sh["v"]).to(w.act_dtype)
    z = normal(sh["z"]).to(w.act_dtype)
    lo, hi = w.log_decay_range
    u = torch.rand(sh["log_decay"], generator=gen, dtype=torch.float32) * (hi - lo) + lo
    log_decay = (-torch.exp(u)).to(gate_dtype)
    beta = torch.sigmoid(normal(sh["beta"])).to(gate_dtype)
    s0 = normal(sh["state"], w.s0_std) if w.s0_std is not None else None
    gn = 1.0 + normal(sh["gn"], 0.1)
    return {"q": q, "k": k, "v": v, "z": z, "log_decay": log_decay, "beta": beta,
            "s0": s0, "gn": gn}
