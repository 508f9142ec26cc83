"""GPU parity with separate key and value head dims (Dk != Dv) and head dims that are not powers
of two (any multiple of 16 up to 128), decode and scan, against the fp64 oracle.  Tolerances as
for the square heads: decode 1e-4, scan 2e-3 (relative to 1 + |oracle|), on y and the final
state.
"""
from __future__ import annotations

import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import make_inputs
from gdn_testutil import DECODE_TOL, SCAN_TOL, oracle_ref, rel_err, small_workload, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


SCAN_CASES = [
    # B, S, Hk, Hv, Dk, Dv, act, head_major
    (1, 40, 1, 2, 64, 128, "bf16", False),    # Dv = 128 over few heads: rows split, cluster norm
    (2, 33, 2, 2, 128, 32, "f16", True),
    (1, 70, 1, 4, 16, 64, "f32", False),
    (1, 50, 1, 1, 128, 64, "bf16", False),
    (2, 20, 1, 2, 32, 128, "f32", False),
    (3, 64, 1, 3, 128, 16, "bf16", True),
    # head dims that are not powers of two (pruned nested prefixes of a 128-wide head)
    (2, 45, 1, 2, 48, 80, "bf16", False),
    (1, 70, 2, 2, 96, 112, "f16", True),
    (2, 33, 1, 3, 112, 48, "f32", False),
    (1, 40, 1, 2, 80, 96, "bf16", True),
    (1, 64, 2, 4, 96, 96, "bf16", False),
    (1, 37, 1, 1, 112, 128, "f16", False),   # Dv = 128 with an odd Dk: the split-head path
]


@pytest.mark.parametrize("case", SCAN_CASES, ids=lambda c: "_".join(map(str, c)))
@pytest.mark.parametrize("gated", [True, False])
def test_scan_rectangular_heads(case, gated):
    B, S, Hk, Hv, Dk, Dv, act, hm = case
    w = small_workload(B=B, S=S, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act=act, head_major=hm,
                       seed=400 + S + Dk + Dv, s0_std=0.05)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                         z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                         head_major=hm)
    torch.cuda.synchronize()
    assert st.shape == (B, Hv, Dv, Dk)
    yr, sr = oracle_ref(inp, gated=gated, head_major=hm)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL


DECODE_CASES = [
    # B, Hk, Hv, Dk, Dv, act
    (3, 1, 2, 64, 128, "bf16"),
    (2, 2, 4, 128, 16, "f16"),
    (4, 1, 1, 32, 64, "f32"),
    (5, 2, 2, 16, 128, "bf16"),
    (3, 1, 2, 48, 80, "bf16"),
    (2, 2, 2, 96, 112, "f16"),
    (4, 1, 3, 112, 48, "f32"),
    (3, 1, 1, 80, 96, "bf16"),
    (2, 1, 2, 128, 96, "bf16"),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "_".join(map(str, c)))
def test_decode_rectangular_heads_several_steps(case):
    B, Hk, Hv, Dk, Dv, act = case
    steps = 4
    w = small_workload(B=B, S=steps, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act=act, seed=500 + Dk + Dv,
                       s0_std=0.05)
    inp = make_inputs(w)
    d = to_dev(inp)
    state = d["s0"].clone()
    ys = []
    for t in range(steps):
        sl = {k: d[k][:, t:t + 1].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
        ys.append(gdn.gdn_decode_step(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"],
                                      state, z=sl["z"], gn=d["gn"]))
    torch.cuda.synchronize()
    yr, sr = oracle_ref(inp)
    assert rel_err(torch.cat(ys, 1), yr) <= DECODE_TOL
    assert rel_err(state, sr) <= DECODE_TOL
