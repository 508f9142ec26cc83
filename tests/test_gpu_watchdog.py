"""Failure detection of the bounded mbarrier waits, on the GPU, without a fault.

gdn_selftest_wait_timeout launches one CTA whose wait expects bytes that no copy sends; the
wait gives up after its time limit, sets the watchdog word and returns.  gdn_device_status must
then report GDN_ERR_TIMEOUT once, clear it, and the context must stay usable.
"""
from __future__ import annotations

import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import make_inputs
from gdn_testutil import DECODE_TOL, oracle_ref, rel_err, small_workload, to_dev

pytestmark = pytest.mark.gpu

GDN_OK, GDN_ERR_TIMEOUT = 0, -9


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


def test_wait_that_runs_out_is_reported_once_and_the_context_stays_usable():
    assert gdn.gdn_device_status() == GDN_OK                # nothing pending before
    assert gdn.gdn_selftest_wait_timeout(5.0) == GDN_OK      # 5 ms limit
    assert gdn.gdn_device_status() == GDN_ERR_TIMEOUT        # reported ...
    assert gdn.gdn_device_status() == GDN_OK                 # ... and cleared
    # a real step afterwards still runs and is correct
    w = small_workload(B=2, S=1, Hk=1, Hv=2, D=128, act="bf16", seed=21, s0_std=0.02)
    inp = make_inputs(w)
    d = to_dev(inp)
    state = d["s0"].clone()
    y = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], state,
                            z=d["z"], gn=d["gn"])
    torch.cuda.synchronize()
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= DECODE_TOL and rel_err(state, sr) <= DECODE_TOL
    assert gdn.gdn_device_status() == GDN_OK


def test_scan_wait_that_runs_out_is_reported_and_the_scan_stays_correct():
    # The chunked scan's own mbarrier waits, with a first-attempt limit of 1 ns: every wait
    # whose barrier is not already complete runs out once, sets the watchdog word and waits
    # again with the full limit, so the scan reports GDN_ERR_TIMEOUT and its results are still
    # right.  With the default limit restored, the next scan reports nothing.
    from gdn_testutil import SCAN_TOL
    w = small_workload(B=1, S=300, Hk=1, Hv=2, D=128, act="bf16", seed=22, s0_std=0.05)
    inp = make_inputs(w)
    d = to_dev(inp)
    yr, sr = oracle_ref(inp)
    assert gdn.gdn_device_status() == GDN_OK
    assert gdn.gdn_selftest_scan_wait_limit(-1.0) == gdn.GDN_ERR_BAD_ARG
    try:
        assert gdn.gdn_selftest_scan_wait_limit(0.001) == GDN_OK
        y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                             z=d["z"], gn=d["gn"], chunked=True)
        torch.cuda.synchronize()
        assert gdn.gdn_device_status() == GDN_ERR_TIMEOUT
        assert gdn.gdn_device_status() == GDN_OK
        assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
    finally:
        assert gdn.gdn_selftest_scan_wait_limit(0.0) == GDN_OK
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                         z=d["z"], gn=d["gn"], chunked=True)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == GDN_OK
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
