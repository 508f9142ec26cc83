"""gdn_scan_split_noalloc through the C ABI: the split scan for callers that cannot allocate
device memory (code inside another framework's memory pool or arena, or where a cudaMalloc is
not allowed), so cannot pass gdn_scan_split a workspace.

The entry point takes its scratch from a fixed device array of the library.  Its results are
checked against gdn_scan_split with a caller workspace, at the scan tolerance, on two calls in a
row (the second call reuses the array the first left behind), and a call whose scratch would
exceed the array is refused on the host.  This file is named to be collected last.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import make_inputs
from gdn_testutil import SCAN_TOL, small_workload, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


def _rel(a: torch.Tensor, ref: torch.Tensor) -> float:
    return float(((a.double() - ref.double()).abs() / (1 + ref.double().abs())).max())


def _inputs(seed: int):
    # one sequence of 8 heads: too few heads to fill the GPU, the case the split is for
    w = small_workload(B=1, S=1500, Hk=2, Hv=8, D=128, act="bf16", seed=seed, s0_std=0.05,
                       ldr=(-6.0, -1.0))
    return to_dev(make_inputs(w))


def _call_noalloc(d, segments, y, state):
    prm = gdn.make_params(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], state, y,
                          z=d["z"], gn=d["gn"], s0=d["s0"])
    lib = gdn.library()
    st = lib.gdn_scan_split_noalloc(ctypes.byref(prm), segments,
                                    torch.cuda.current_stream().cuda_stream)
    return st, prm


def test_noalloc_split_matches_the_workspace_split_on_two_calls_in_a_row():
    segments = 4
    for seed in (901, 902):
        d = _inputs(seed)
        args = (d["q"], d["k"], d["v"], d["log_decay"], d["beta"])
        y_ref, s_ref = gdn.gdn_scan_split(*args, s0=d["s0"], z=d["z"], gn=d["gn"],
                                          segments=segments)
        prm = gdn.make_params(*args, s_ref, y_ref, z=d["z"], gn=d["gn"], s0=d["s0"])
        assert 0 < gdn.gdn_scan_split_workspace(prm, segments) <= \
            gdn.GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES
        y = torch.full_like(y_ref, float("nan"))
        state = torch.full_like(s_ref, float("nan"))
        st, _ = _call_noalloc(d, segments, y, state)
        assert st == gdn.GDN_OK, gdn.gdn_last_error()
        torch.cuda.synchronize()
        assert gdn.gdn_device_status() == gdn.GDN_OK
        assert _rel(y, y_ref) <= SCAN_TOL, seed
        assert _rel(state, s_ref) <= SCAN_TOL, seed


def test_noalloc_split_refuses_scratch_beyond_its_fixed_size():
    # 8 sequences of 8 heads in 8 segments: 88 MiB of scratch, more than the fixed 16 MiB
    w = small_workload(B=8, S=64, Hk=2, Hv=8, D=128, act="bf16", seed=903, s0_std=0.05)
    d = to_dev(make_inputs(w))
    y = torch.full(d["v"].shape, 7.0, dtype=torch.float32, device="cuda")
    state = torch.full(d["s0"].shape, 7.0, dtype=torch.float32, device="cuda")
    st, prm = _call_noalloc(d, 8, y, state)
    assert gdn.gdn_scan_split_workspace(prm, 8) > gdn.GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES
    assert st == gdn.GDN_ERR_BAD_ARG
    assert "exceeds" in gdn.gdn_last_error()
    torch.cuda.synchronize()
    assert bool(torch.all(y == 7.0)) and bool(torch.all(state == 7.0))   # nothing enqueued
