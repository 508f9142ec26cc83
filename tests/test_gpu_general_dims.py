"""GPU parity for head dims the tiled kernels do not take: any Dk, Dv up to 256 that are not
multiples of 16 (pruned nested-prefix widths of modelopt puzzletron.pruning.gated_delta_net,
slice_gated_delta_net_state_dict / GDNShape, can be any size).  Those run the general kernel
(f32 on CUDA cores, the head's memory in shared memory), for the decode step and the scan, and
gdn_scan_split runs the whole sequence in one launch there.  Against the fp64 oracle at the
usual tolerances (decode 1e-4, scan 2e-3, relative to 1 + |oracle|) on y and the final state;
the f32 arithmetic keeps the scan far inside its bar, which is checked too.
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


CASES = [
    # B, S, Hk, Hv, Dk, Dv, act, head_major
    (1, 37, 1, 2, 100, 72, "bf16", False),
    (2, 20, 2, 4, 24, 40, "f16", True),
    (1, 25, 1, 1, 128, 120, "f32", False),
    (1, 9, 1, 2, 1, 1, "f32", False),          # the smallest head
    (2, 11, 1, 3, 5, 7, "bf16", False),
    (1, 70, 2, 2, 17, 129, "f16", False),      # Dv above 128, not a multiple of 16
    (1, 6, 1, 2, 232, 232, "bf16", True),      # the largest square head the kernel keeps
    (1, 12, 1, 1, 255, 9, "f32", False),
    (1, 30, 1, 2, 48, 100, "bf16", False),     # one dim tiled, the other not
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c)))
@pytest.mark.parametrize("gated", [True, False], ids=["gated", "raw_o"])
def test_general_dims_scan_matches_oracle(case, gated):
    B, S, Hk, Hv, Dk, Dv, act, hm = case
    w = small_workload(B=B, S=S, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act=act, head_major=hm,
                       seed=700 + Dk + Dv, s0_std=0.1)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                         z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                         head_major=hm)
    torch.cuda.synchronize()
    yr, sr = oracle_ref(inp, gated=gated, head_major=hm)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
    assert rel_err(y, yr) <= 1e-4 and rel_err(st, sr) <= 1e-4      # f32 throughout


@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c)))
def test_general_dims_decode_matches_oracle(case):
    B, _, Hk, Hv, Dk, Dv, act, hm = case
    w = small_workload(B=B, S=1, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act=act, head_major=hm,
                       seed=800 + Dk + Dv, s0_std=0.1)
    inp = make_inputs(w)
    d = to_dev(inp)
    state = d["s0"].clone()
    y = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], state,
                            z=d["z"], gn=d["gn"], head_major=hm)
    torch.cuda.synchronize()
    yr, sr = oracle_ref(inp, head_major=hm)
    assert rel_err(y, yr) <= DECODE_TOL and rel_err(state, sr) <= DECODE_TOL


def test_general_dims_zero_state_gates_in_act_dtype_and_in_place_resume():
    w = small_workload(B=2, S=40, Hk=1, Hv=2, Dk=36, Dv=44, act="bf16", seed=901, s0_std=None)
    inp = make_inputs(w, gate_dtype=torch.bfloat16)
    d = to_dev(inp)
    y0, s0 = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=None,
                          z=d["z"], gn=d["gn"])
    yr, sr = oracle_ref(inp, s0=None)
    assert rel_err(y0, yr) <= 1e-4 and rel_err(s0, sr) <= 1e-4
    # two calls, the second resuming in place from the first's memory
    state = torch.zeros(2, 2, 44, 36, device="cuda")
    parts = []
    for a, b in ((0, 15), (15, 40)):
        sl = {k: d[k][:, a:b].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
        yp, _ = gdn.gdn_scan(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"], state,
                             s0=state, z=sl["z"], gn=d["gn"])
        parts.append(yp)
    torch.cuda.synchronize()
    assert rel_err(torch.cat(parts, 1), yr) <= 1e-4 and rel_err(state, sr) <= 1e-4


def test_general_dims_split_runs_the_whole_sequence():
    w = small_workload(B=1, S=90, Hk=1, Hv=2, Dk=20, Dv=28, act="f16", seed=902, s0_std=0.1)
    inp = make_inputs(w)
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["log_decay"], d["beta"])
    prm = gdn.make_params(*args, torch.empty(1, 2, 28, 20, device="cuda"),
                          torch.empty(d["v"].shape, device="cuda"), z=d["z"], gn=d["gn"],
                          s0=d["s0"])
    assert gdn.gdn_scan_split_workspace(prm, 4) == 0
    y0, s0 = gdn.gdn_scan(*args, s0=d["s0"], z=d["z"], gn=d["gn"])
    y1, s1 = gdn.gdn_scan_split(*args, s0=d["s0"], z=d["z"], gn=d["gn"], segments=4)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(s0, s1)


def test_general_dims_many_heads():
    # more heads than SMs, grouped keys
    w = small_workload(B=3, S=5, Hk=20, Hv=80, Dk=40, Dv=24, act="f16", seed=903, s0_std=0.1)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                         z=d["z"], gn=d["gn"])
    torch.cuda.synchronize()
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= 1e-4 and rel_err(st, sr) <= 1e-4


def test_general_dims_host_fed_decode():
    # GDN_FLAG_HOST_IO: the general kernel reads the inputs from pinned host memory and writes y
    # there with plain loads and stores
    w = small_workload(B=3, S=1, Hk=1, Hv=2, Dk=36, Dv=20, act="bf16", seed=904, s0_std=0.1)
    inp = make_inputs(w)
    host = {k: inp[k].contiguous().pin_memory()
            for k in ("q", "k", "v", "z", "log_decay", "beta")}
    state = inp["s0"].cuda()
    y = gdn.gdn_decode_step(host["q"], host["k"], host["v"], host["log_decay"], host["beta"],
                            state, z=host["z"], gn=inp["gn"].cuda(), host_io=True)
    torch.cuda.synchronize()
    assert not y.is_cuda
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= DECODE_TOL and rel_err(state, sr) <= DECODE_TOL


@pytest.mark.parametrize("Dk,Dv,B,Hv", [(40, 24, 8, 96), (200, 196, 2, 100), (9, 7, 4, 64)],
                         ids=["small_heads", "large_heads", "scalar_copies"])
def test_general_dims_decode_many_heads(Dk, Dv, B, Hv):
    # the general decode kernel over many heads: several resident per SM (small memories), one
    # per SM in waves (large), and the memory by 4-byte copies (Dv Dk not a multiple of 4)
    w = small_workload(B=B, S=1, Hk=Hv // 4, Hv=Hv, Dk=Dk, Dv=Dv, act="bf16", seed=905 + Dk,
                       s0_std=0.1)
    inp = make_inputs(w)
    d = to_dev(inp)
    state = d["s0"].clone()
    y = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], state,
                            z=d["z"], gn=d["gn"])
    torch.cuda.synchronize()
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= DECODE_TOL and rel_err(state, sr) <= DECODE_TOL
