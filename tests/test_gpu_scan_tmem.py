"""GPU parity of the tensor-memory chunked scan (gdn_scan with GDN_FLAG_SCAN_TMEM) against the
fp64 oracle, through the C ABI.

The kernel applies to bf16 activations with Dk = Dv = 128; it processes 32-token chunks, keeps
a deferred decay scale that it folds into the memory when it would underflow, and looks one
chunk ahead.  The cases below cross the chunk boundary (S = 31..33, 63..65), run many chunks
(with and without folds), vary GQA, layout, gating and the initial state, and check that other
shapes with the flag set run the default kernel.  Tolerance as for every scan:
max |gpu - oracle| / (1 + |oracle|) <= 2e-3 on y and on the final state.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import PREFILL_B4, make_inputs
from gdn_testutil import (SCAN_TOL, guard_intact, guarded, oracle_ref, record_margin, rel_err,
                          small_workload, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


def run_tmem(inp, *, gated=True, head_major=False, s0="inp"):
    d = to_dev(inp)
    s0v = d["s0"] if s0 == "inp" else s0
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=s0v,
                         z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                         head_major=head_major, tmem=True)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    return y, st


CASES = [
    # B, S, Hk, Hv, head_major
    (1, 1, 1, 1, False),
    (2, 5, 2, 4, False),
    (1, 31, 1, 2, True),
    (1, 32, 2, 2, False),
    (2, 33, 2, 4, True),
    (1, 63, 1, 4, False),
    (1, 65, 4, 4, True),
    (2, 100, 8, 32, False),
    (1, 130, 16, 64, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c)))
@pytest.mark.parametrize("gated", [True, False])
def test_tmem_scan_edge_shapes(case, gated):
    B, S, Hk, Hv, hm = case
    w = small_workload(B=B, S=S, Hk=Hk, Hv=Hv, D=128, act="bf16", head_major=hm,
                       seed=700 + S + Hv, s0_std=0.2)
    inp = make_inputs(w)
    y, st = run_tmem(inp, gated=gated, head_major=hm)
    yr, sr = oracle_ref(inp, gated=gated, head_major=hm)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
    if not gated:
        # no norm amplification: the split-bf16 products reach about 1e-6
        assert rel_err(y, yr) <= 1e-4


@pytest.mark.parametrize("ldr", [(-0.1, 0.0), (-3.0, 0.0), (-8.0, -3.0)],
                         ids=["slow_decay", "fast_decay_folds", "near_one"])
def test_tmem_scan_many_chunks(ldr):
    # 20 chunks: the staging ring wraps five times; with fast decay the deferred decay scale
    # underflows and is folded into the memory every few chunks
    w = small_workload(B=1, S=640, Hk=2, Hv=4, D=128, act="bf16", seed=711, s0_std=0.05,
                       ldr=ldr)
    inp = make_inputs(w)
    y, st = run_tmem(inp)
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
    # every chunk is right, not only the end state
    err = np.abs(y.detach().cpu().double().numpy() - yr) / (1 + np.abs(yr))
    per_chunk = [float(err[:, c:c + 32].max()) for c in range(0, 640, 32)]
    assert max(per_chunk) <= SCAN_TOL, per_chunk


def test_tmem_scan_zero_state_and_in_place_resume():
    w = small_workload(B=2, S=90, Hk=2, Hv=4, D=128, act="bf16", s0_std=None, seed=712)
    inp = make_inputs(w)
    y0, s0 = run_tmem(inp, s0=None)
    yr, sr = oracle_ref(inp, s0=None)
    assert rel_err(y0, yr) <= SCAN_TOL and rel_err(s0, sr) <= SCAN_TOL
    # resume in place from the state after the first 40 tokens
    d = to_dev(inp)
    state = torch.zeros(2, 4, 128, 128, device="cuda")
    ys = []
    for a, b in ((0, 40), (40, 90)):
        sl = {k: d[k][:, a:b].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
        yp, _ = gdn.gdn_scan(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"], state,
                             s0=state, z=sl["z"], gn=d["gn"], tmem=True)
        ys.append(yp)
    torch.cuda.synchronize()
    assert rel_err(torch.cat(ys, dim=1), yr) <= SCAN_TOL and rel_err(state, sr) <= SCAN_TOL


def test_tmem_scan_matches_default_kernel():
    w = small_workload(B=2, S=200, Hk=4, Hv=8, D=128, act="bf16", seed=713, s0_std=0.1)
    inp = make_inputs(w)
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["log_decay"], d["beta"])
    y1, s1 = gdn.gdn_scan(*args, s0=d["s0"], z=d["z"], gn=d["gn"], tmem=True)
    y2, s2 = gdn.gdn_scan(*args, s0=d["s0"], z=d["z"], gn=d["gn"])
    torch.cuda.synchronize()
    scale = 1 + y2.abs()
    assert float(((y1 - y2).abs() / scale).max()) <= SCAN_TOL
    assert float(((s1 - s2).abs() / (1 + s2.abs())).max()) <= SCAN_TOL


@pytest.mark.parametrize("act,D", [("f16", 128), ("bf16", 64), ("f32", 128)])
def test_tmem_flag_on_other_shapes_runs_the_default_kernel(act, D):
    w = small_workload(B=1, S=40, Hk=1, Hv=2, D=D, act=act, seed=714, s0_std=0.1)
    inp = make_inputs(w)
    y, st = run_tmem(inp)
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL


@pytest.mark.parametrize("gated", [True, False], ids=["gated", "raw_o"])
def test_tmem_scan_full_size_prefill(gated):
    w = PREFILL_B4
    inp = make_inputs(w)
    d = to_dev(inp)
    y, ywhole = guarded(tuple(d["v"].shape))
    st, swhole = guarded((w.B, w.Hv, w.Dv, w.Dk))
    gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st, y, s0=d["s0"],
                 z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                 head_major=w.head_major, tmem=True)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    del d
    yr, sr = oracle_ref(inp, gated=gated, head_major=w.head_major)
    ey, es = rel_err(y, yr), rel_err(st, sr)
    record_margin(w.name, "gdn_scan tensor-memory (GDN_FLAG_SCAN_TMEM)",
                  "gated y" if gated else "raw o", ey, es, SCAN_TOL)
    assert ey <= SCAN_TOL and es <= SCAN_TOL
    assert guard_intact(ywhole, y.numel()) and guard_intact(swhole, st.numel())
