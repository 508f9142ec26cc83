"""GPU parity with separate key and value head dims (Dk != Dv), head dims that are not powers
of two (any multiple of 16 up to 128) and head dims of 256, decode and scan, against the fp64
oracle.  Tolerances as for the square heads: decode 1e-4, scan 2e-3 (relative to 1 + |oracle|),
on y and the final state.

A head dim of 256 takes other paths: the scan runs at most 4 row warps per CTA when Dk = 256
(a head's rows then spread over a cluster of 2 to 8 CTAs), reads f32 k, q rows of 256 straight
from global memory, and takes 128 rows per CTA when Dv = 256; the decode step cuts a head of
more than 64 KB of state into row blocks that one CTA runs back to back.
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
    (1, 40, 1, 2, 128, 112, "f32", False),   # 7 row warps of f32 rows do not fit: 7 CTAs
    # head dims of 256
    (1, 40, 1, 2, 256, 256, "bf16", False),   # 4 row warps, a cluster of 4 CTAs per head
    (2, 33, 1, 2, 256, 128, "f16", True),
    (1, 37, 1, 1, 256, 256, "f32", False),    # f32 k, q rows read from global memory
    (1, 45, 1, 2, 128, 256, "bf16", False),
    (2, 35, 1, 2, 64, 256, "f16", True),
    (1, 33, 1, 2, 256, 80, "bf16", False),    # 1 row warp, a cluster of 5
    (1, 50, 1, 1, 256, 112, "f32", True),     # a cluster of 7
    (1, 40, 1, 2, 256, 96, "f16", False),     # 3 row warps, a cluster of 2
    (2, 20, 1, 2, 256, 32, "bf16", False),
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
    # head dims of 256
    (3, 1, 2, 256, 256, "bf16"),     # 4 row blocks of 64 rows per head
    (2, 1, 2, 256, 128, "f32"),
    (2, 2, 2, 128, 256, "f16"),      # 2 row blocks of 128 rows
    (3, 1, 3, 256, 80, "bf16"),      # 5 row blocks of 16 rows
    (2, 1, 2, 256, 48, "f16"),       # a whole head of 48 x 256
    (2, 1, 2, 256, 96, "f32"),
    (2, 1, 1, 112, 256, "bf16"),
    (2, 1, 2, 64, 256, "bf16"),
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


@pytest.mark.parametrize("dims,heads", [((256, 256), (20, 1, 16)), ((256, 80), (32, 2, 32)),
                                        ((128, 256), (24, 2, 8))],
                         ids=["256x256", "256x80", "128x256"])
@pytest.mark.parametrize("gated", [True, False])
def test_decode_head_dim_256_many_heads(dims, heads, gated):
    # more heads than resident CTAs: every CTA runs several heads of several row blocks, so the
    # per-head norm sum and the gates of the next head carry over correctly
    Dk, Dv = dims
    B, Hk, Hv = heads
    steps = 2
    w = small_workload(B=B, S=steps, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act="bf16", seed=520 + Dv,
                       s0_std=0.05)
    inp = make_inputs(w)
    d = to_dev(inp)
    state = d["s0"].clone()
    ys = []
    for t in range(steps):
        sl = {k: d[k][:, t:t + 1].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
        ys.append(gdn.gdn_decode_step(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"],
                                      state, z=sl["z"] if gated else None,
                                      gn=d["gn"] if gated else None))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    yr, sr = oracle_ref(inp, gated=gated)
    assert rel_err(torch.cat(ys, 1), yr) <= DECODE_TOL
    assert rel_err(state, sr) <= DECODE_TOL


def test_scan_head_dim_256_many_heads():
    # more CTAs than fit on the device at once for Dk = Dv = 256 (4 per head)
    w = small_workload(B=4, S=70, Hk=4, Hv=16, Dk=256, Dv=256, act="bf16", seed=530,
                       s0_std=0.05)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                         z=d["z"], gn=d["gn"])
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
