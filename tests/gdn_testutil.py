"""Shared helpers of the GPU parity tests (device moves, oracle calls, error measures)."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from linear_attention_recurrence_gdn_gb300.workloads import TINY, Workload, make_inputs

# Elementwise tolerances on y and the final state:  max |gpu - ref| / (1 + |ref|).
DECODE_TOL = 1e-4
SCAN_TOL = 2e-3

CPUS = os.cpu_count() or 1

# Where the full-size parity tests append their measured margins (JSON lines); unset: only
# printed.  tests/parity_table.py turns such a file into the margin table under profiles/.
PARITY_LOG = os.environ.get("GDN_PARITY_LOG")


def small_workload(B=1, S=4, Hk=1, Hv=2, D=16, act="f32", head_major=False, s0_std=0.1,
                   seed=5, ldr=(-3.0, 0.0), Dk=None, Dv=None) -> Workload:
    return TINY.replace(name="case", B=B, S=S, Hk=Hk, Hv=Hv, Dk=Dk or D, Dv=Dv or D, act=act,
                        head_major=head_major, s0_std=s0_std, seed=seed,
                        log_decay_range=ldr)


def to_dev(inp: dict, dev="cuda") -> dict:
    return {k: (None if v is None else v.to(dev).contiguous()) for k, v in inp.items()}


def oracle_ref(inp: dict, *, gated=True, head_major=False, heads=None, s0="inp"):
    s0v = inp["s0"] if s0 == "inp" else s0
    return oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                      z=inp["z"] if gated else None, gn=inp["gn"] if gated else None,
                      s0=s0v, head_major=head_major, heads=heads, threads=CPUS)


def rel_err(gpu: torch.Tensor, ref: np.ndarray, mask=None) -> float:
    a = gpu.detach().cpu().double().numpy()
    if mask is not None:
        a, ref = a[mask], ref[mask]
    if ref.size == 0:
        return 0.0
    assert np.all(np.isfinite(a)), "non-finite GPU output"
    return float(np.max(np.abs(a - ref) / (1.0 + np.abs(ref))))


def record_margin(workload: str, kernel: str, output: str, err_y: float, err_state: float,
                  tol: float):
    """Record a parity case's max |gpu - oracle| / (1 + |oracle|) on y and on the final state
    next to its tolerance (printed, and appended to $GDN_PARITY_LOG when set)."""
    rec = {"workload": workload, "kernel": kernel, "output": output, "err_y": err_y,
           "err_state": err_state, "tol": tol}
    print("parity-margin", json.dumps(rec))
    if PARITY_LOG:
        with open(PARITY_LOG, "a") as f:
            f.write(json.dumps(rec) + "\n")


def guarded(shape, dtype=torch.float32, dev="cuda", fill=1234.5, guard=4096):
    """A tensor with `guard` sentinel elements on both sides inside one allocation.

    Returns (view, whole); check_guard(whole, view) verifies the sentinels are untouched.
    """
    n = int(np.prod(shape))
    whole = torch.full((n + 2 * guard,), fill, dtype=dtype, device=dev)
    view = whole[guard:guard + n].view(shape)
    return view, whole


def guard_intact(whole: torch.Tensor, n: int, guard=4096, fill=1234.5) -> bool:
    w = whole.detach().cpu()
    return bool(torch.all(w[:guard] == fill)) and bool(torch.all(w[guard + n:] == fill))


__all__ = ["DECODE_TOL", "SCAN_TOL", "small_workload", "to_dev", "oracle_ref", "rel_err",
           "guarded", "guard_intact", "make_inputs", "record_margin"]
