"""GPU parity of gdn_scan_split (the sequence cut into segments that run in parallel) against
the fp64 oracle, through the C ABI.

The page's update is affine in the memory (logicaffeine codegen_cuda::gdn, "The fusion"), so
a segment maps its start memory S0 to S0 M + N.  The split scan computes M and N per segment,
composes the start memories, and reruns each segment from its start.  The cases cross
segment boundaries inside and between 32-token chunks, use more segments than tokens, both
layouts, grouped heads, Dk != Dv, heads of 256, gated and raw outputs, with and without s0,
and the in-place resume.  Tolerance as for every scan: 2e-3 relative to 1 + |oracle|.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import LONG_B2, make_inputs
from gdn_testutil import SCAN_TOL, oracle_ref, record_margin, rel_err, small_workload, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


CASES = [
    # B, S, Hk, Hv, Dk, Dv, act, head_major, segments, gated, with s0
    (1, 100, 1, 2, 128, 128, "bf16", False, 3, True, True),
    (2, 257, 2, 4, 64, 128, "f16", True, 4, False, False),
    (1, 64, 1, 1, 128, 128, "f32", False, 2, True, True),
    (1, 1000, 1, 2, 128, 128, "bf16", False, 7, True, True),
    (1, 40, 1, 2, 32, 48, "bf16", True, 5, True, True),
    (2, 70, 1, 2, 256, 256, "bf16", False, 2, True, True),
    (1, 33, 1, 2, 128, 128, "bf16", False, 40, True, True),    # more segments than tokens
    (3, 90, 1, 3, 128, 64, "f16", False, 3, True, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c)))
def test_split_scan_matches_oracle(case):
    B, S, Hk, Hv, Dk, Dv, act, hm, nseg, gated, with_s0 = case
    w = small_workload(B=B, S=S, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act=act, head_major=hm,
                       seed=800 + S + nseg, s0_std=0.05 if with_s0 else None)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = gdn.gdn_scan_split(d["q"], d["k"], d["v"], d["log_decay"], d["beta"],
                               s0=d["s0"], z=d["z"] if gated else None,
                               gn=d["gn"] if gated else None, head_major=hm, segments=nseg)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    yr, sr = oracle_ref(inp, gated=gated, head_major=hm)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL


def test_split_scan_fast_decay_and_in_place_resume():
    # decay fast enough that the deferred scale folds inside every segment; s0 is state
    w = small_workload(B=1, S=600, Hk=2, Hv=4, D=128, act="bf16", seed=811, s0_std=0.1,
                       ldr=(-3.0, 0.0))
    inp = make_inputs(w)
    d = to_dev(inp)
    state = d["s0"].clone()
    y, st = gdn.gdn_scan_split(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], state,
                               s0=state, z=d["z"], gn=d["gn"], segments=6)
    torch.cuda.synchronize()
    assert st.data_ptr() == state.data_ptr()
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(state, sr) <= SCAN_TOL


def test_split_scan_agrees_with_scan_and_one_segment_is_the_scan():
    w = small_workload(B=2, S=200, Hk=2, Hv=4, D=128, act="bf16", seed=812, s0_std=0.05)
    inp = make_inputs(w)
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["log_decay"], d["beta"])
    y0, s0 = gdn.gdn_scan(*args, s0=d["s0"], z=d["z"], gn=d["gn"])
    y1, s1 = gdn.gdn_scan_split(*args, s0=d["s0"], z=d["z"], gn=d["gn"], segments=1)
    y4, s4 = gdn.gdn_scan_split(*args, s0=d["s0"], z=d["z"], gn=d["gn"], segments=4)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(s0, s1)      # the same kernel launch
    scale = 1 + y0.abs()
    assert float(((y4 - y0).abs() / scale).max()) <= SCAN_TOL
    assert float(((s4 - s0).abs() / (1 + s0.abs())).max()) <= SCAN_TOL


def test_split_workspace_size_formula():
    w = small_workload(B=3, S=100, Hk=1, Hv=2, Dk=64, Dv=128, act="bf16", seed=813)
    d = to_dev(make_inputs(w))
    y = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
    st = torch.empty(3, 2, 128, 64, device="cuda")
    prm = gdn.make_params(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st, y)
    bh = 3 * 2
    for nseg, g in ((1, 1), (2, 2), (3, 3), (7, 7), (60, 50), (100, 100), (1000, 100)):
        need = gdn.gdn_scan_split_workspace(prm, nseg)
        expect = 0 if g == 1 else 4 * ((g - 1) * bh * 64 * 64 + (g - 1) * bh * 128 * 64
                                       + g * bh * 128 * 64)
        assert need == expect, (nseg, need, expect)


@pytest.mark.parametrize("nseg", [4, 8])
def test_split_scan_long_slow_decay_few_heads(nseg):
    # the regime the split is built and measured for: one sequence of 16384 f16 tokens with 8
    # value heads and the long workload's slow decay (alpha up to 0.9997), where the f32
    # composition S0 M + N runs over many near-identity transitions
    w = LONG_B2.replace(name="long_f16_b1_s16384_hk2_hv8_d128", B=1, Hk=2, Hv=8)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = gdn.gdn_scan_split(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                               z=d["z"], gn=d["gn"], segments=nseg)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    del d
    yr, sr = oracle_ref(inp)
    ey, es = rel_err(y, yr), rel_err(st, sr)
    record_margin(w.name, f"gdn_scan_split, {nseg} segments", "gated y", ey, es, SCAN_TOL)
    assert ey <= SCAN_TOL and es <= SCAN_TOL


def test_split_one_grid_and_two_launches_agree_around_the_threshold():
    # With Dk == Dv the transitions and offsets share one grid while their 2 (g - 1) B Hv
    # (segment, head) pairs fit in half the SMs, else they run as two launches.  One shape on
    # each side of that threshold, from this device's SM count: both paths against the oracle.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    g = 3                                              # segments: 2 (g - 1) = 4 pairs per head
    bh_under = (sms // 2) // (2 * (g - 1))             # largest B Hv on the one-grid side
    results = []
    for bh in (bh_under, bh_under + 1):
        B, Hv = bh, 1
        w = small_workload(B=B, S=96, Hk=1, Hv=Hv, D=64, act="bf16", seed=820 + bh,
                           s0_std=0.05)
        inp = make_inputs(w)
        d = to_dev(inp)
        y, st = gdn.gdn_scan_split(d["q"], d["k"], d["v"], d["log_decay"], d["beta"],
                                   s0=d["s0"], z=d["z"], gn=d["gn"], segments=g)
        torch.cuda.synchronize()
        yr, sr = oracle_ref(inp)
        assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
        results.append(2 * (g - 1) * B * Hv <= sms // 2)
    assert results == [True, False]                    # one case on each side


def test_split_scan_on_a_side_stream_keeps_its_own_workspace():
    # The binding allocates the workspace on the current stream; the kernels run on a side
    # stream.  Memory allocated and filled on the current stream right after the call must not
    # receive the freed workspace block while the side stream still uses it.
    w = small_workload(B=1, S=2000, Hk=2, Hv=4, D=128, act="bf16", seed=830, s0_std=0.05)
    inp = make_inputs(w)
    d = to_dev(inp)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        y = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
        st = torch.empty(d["s0"].shape, dtype=torch.float32, device="cuda")
    y.record_stream(side)
    st.record_stream(side)
    gdn.gdn_scan_split(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st, y, s0=d["s0"],
                       z=d["z"], gn=d["gn"], segments=4, stream=side)
    junk = [torch.full((1 << 20,), 3.0e4, device="cuda") for _ in range(8)]
    torch.cuda.synchronize()
    del junk
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
