"""GPU parity of gdn_decode_step against the fp64 oracle (through the C ABI).

Tolerance: max |gpu - oracle| / (1 + |oracle|) <= 1e-4 on y and on the updated state, for
the f32-accumulated decode step.  Every case compares both outputs: a kernel that ignored
the memory would otherwise pass (logicaffeine codegen_cuda::gdn, emit_gated_delta_forward
prints O and the mutated S for that reason).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import (DECODE_B64, DECODE_B256_HM, TINY,
                                                             make_inputs)
from gdn_testutil import (DECODE_TOL, guard_intact, guarded, oracle_ref, record_margin, rel_err,
                          small_workload, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


def run_decode(inp, *, gated=True, head_major=False, state=None):
    d = to_dev(inp)
    st = d["s0"].clone() if state is None else state
    y = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st,
                            z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                            head_major=head_major)
    torch.cuda.synchronize()
    return y, st


@pytest.mark.parametrize("gated", [True, False], ids=["gated", "raw_o"])
@pytest.mark.parametrize("w", [DECODE_B64, DECODE_B256_HM], ids=lambda w: w.name)
def test_full_size_decode_matches_oracle(w, gated):
    # raw o as well: rmsnorm hides a missing 1/sqrt(Dk) or alpha on o; the raw output does not
    inp = make_inputs(w)
    d = to_dev(inp)
    state, whole = guarded(tuple(d["s0"].shape))
    state.copy_(d["s0"])
    y, ywhole = guarded(tuple(d["v"].shape))
    gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], state, y,
                        z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                        head_major=w.head_major)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    yr, sr = oracle_ref(inp, gated=gated, head_major=w.head_major)
    ey, es = rel_err(y, yr), rel_err(state, sr)
    record_margin(w.name, "gdn_decode_step", "gated y" if gated else "raw o", ey, es,
                  DECODE_TOL)
    assert ey <= DECODE_TOL
    assert es <= DECODE_TOL
    assert guard_intact(whole, state.numel()) and guard_intact(ywhole, y.numel())


def test_tiny_workload_as_eight_decode_steps():
    inp = make_inputs(TINY)
    d = to_dev(inp)
    state = d["s0"].clone()
    ys = []
    for t in range(TINY.S):
        sl = {k: d[k][:, t:t + 1].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
        ys.append(gdn.gdn_decode_step(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"],
                                      state, z=sl["z"], gn=d["gn"]))
    torch.cuda.synchronize()
    yr, sr = oracle_ref(inp)
    assert rel_err(torch.cat(ys, 1), yr) <= DECODE_TOL
    assert rel_err(state, sr) <= DECODE_TOL


@pytest.mark.parametrize("head_major,gated,act", [(False, True, "bf16"), (True, True, "f16"),
                                                   (False, False, "f32")])
def test_host_decode_step_over_several_steps(head_major, gated, act):
    # HostDecodeStep: the kernel reads the step's inputs from pinned host memory and writes y
    # to pinned host memory (GDN_FLAG_HOST_IO) on the device-resident state; every step writes
    # new inputs into the host views, which the next call must read
    steps = 5
    w = small_workload(B=3, S=steps, Hk=2, Hv=4, D=128, act=act, head_major=head_major,
                       seed=640, s0_std=0.05)
    inp = make_inputs(w)
    names = ["q", "k", "v", "log_decay", "beta"] + (["z"] if gated else [])
    tdim = 2 if head_major else 1                          # the token axis
    step_in = lambda t: {n: inp[n].narrow(tdim, t, 1).contiguous() for n in names}
    s0 = inp["s0"].to("cuda")
    state = s0.clone()
    gn = inp["gn"].to("cuda") if gated else None
    stepper = gdn.HostDecodeStep(step_in(0), state, gn, head_major=head_major)
    torch.cuda.synchronize()
    assert torch.equal(state, s0)                          # construction runs no step
    assert stepper.h2d_bytes == sum(t.numel() * t.element_size() for t in step_in(0).values())
    ys = []
    for t in range(steps):
        for n, x in step_in(t).items():
            stepper.host[n].copy_(x)
        ys.append(stepper.run().clone())
    yr, sr = oracle_ref(inp, gated=gated, head_major=head_major)
    # the stepper keeps the tensors its graph points at alive
    assert stepper.state is state and stepper.gn is gn
    assert rel_err(torch.cat(ys, tdim), yr) <= DECODE_TOL
    assert rel_err(state, sr) <= DECODE_TOL


def test_host_decode_step_on_its_own_stream():
    # a stepper bound to a side stream, and one step on another stream named in run()
    steps = 3
    w = small_workload(B=2, S=steps, Hk=2, Hv=4, D=128, act="bf16", seed=660, s0_std=0.05)
    inp = make_inputs(w)
    names = ["q", "k", "v", "log_decay", "beta", "z"]
    step_in = lambda t: {n: inp[n].narrow(1, t, 1).contiguous() for n in names}
    state = inp["s0"].to("cuda")
    gn = inp["gn"].to("cuda")
    side, other = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    stepper = gdn.HostDecodeStep(step_in(0), state, gn, stream=side)
    ys = []
    for t in range(steps):
        for n, x in step_in(t).items():
            stepper.host[n].copy_(x)
        ys.append(stepper.run(stream=other if t == 1 else None).clone())
    yr, sr = oracle_ref(inp)
    assert rel_err(torch.cat(ys, 1), yr) <= DECODE_TOL
    assert rel_err(state, sr) <= DECODE_TOL


@pytest.mark.parametrize("placement", ["inputs_host", "y_host", "all_host"])
@pytest.mark.parametrize("dims", [(128, 128), (64, 256), (256, 80)], ids=lambda d: f"{d[0]}x{d[1]}")
def test_decode_host_io_placements(placement, dims):
    # GDN_FLAG_HOST_IO accepts pinned host memory and device memory in any mix; several steps,
    # including heads cut into row blocks (Dv = 256 with Dk = 64 is one 64 KB unit; Dk = 256,
    # Dv = 80 five units of 16 rows)
    Dk, Dv = dims
    steps = 3
    w = small_workload(B=5, S=steps, Hk=2, Hv=4, Dk=Dk, Dv=Dv, act="bf16", seed=650 + Dv,
                       s0_std=0.05)
    inp = make_inputs(w)
    state = inp["s0"].to("cuda")
    gn = inp["gn"].to("cuda")
    host_in = placement in ("inputs_host", "all_host")
    host_y = placement in ("y_host", "all_host")
    ys = []
    for t in range(steps):
        sl = {n: inp[n][:, t:t + 1].contiguous() for n in ("q", "k", "v", "z", "log_decay", "beta")}
        sl = {n: (x.pin_memory() if host_in else x.to("cuda")) for n, x in sl.items()}
        y = (torch.empty(sl["v"].shape, dtype=torch.float32).pin_memory() if host_y
             else torch.empty(sl["v"].shape, dtype=torch.float32, device="cuda"))
        gdn.gdn_decode_step(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"], state, y,
                            z=sl["z"], gn=gn, host_io=True)
        torch.cuda.synchronize()
        ys.append(y.cpu().clone())
    yr, sr = oracle_ref(inp)
    assert rel_err(torch.cat(ys, 1), yr) <= DECODE_TOL
    assert rel_err(state, sr) <= DECODE_TOL


def test_decode_host_io_many_heads_matches_device_path():
    # every CTA runs several heads: the pieces staged one unit ahead must follow the heads of
    # a CTA's range; bit-identical to the device-memory path (same kernel arithmetic)
    w = DECODE_B64.replace(B=20)
    inp = make_inputs(w)
    d = to_dev(inp)
    st_dev = d["s0"].clone()
    y_dev = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st_dev,
                                z=d["z"], gn=d["gn"])
    h = {n: inp[n].contiguous().pin_memory() for n in ("q", "k", "v", "z", "log_decay", "beta")}
    st_host = d["s0"].clone()
    y_host = gdn.gdn_decode_step(h["q"], h["k"], h["v"], h["log_decay"], h["beta"], st_host,
                                 z=h["z"], gn=d["gn"], host_io=True)
    torch.cuda.synchronize()
    assert not y_host.is_cuda and y_host.is_pinned()
    assert torch.equal(y_host, y_dev.cpu()) and torch.equal(st_host, st_dev)


SHAPES = [(D, Hk, Hv) for D in (16, 32, 64, 128) for (Hk, Hv) in ((2, 2), (2, 4), (1, 4))]


@pytest.mark.parametrize("act", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"D{s[0]}_Hk{s[1]}_Hv{s[2]}")
@pytest.mark.parametrize("gated", [True, False])
def test_decode_shapes_and_dtypes(act, shape, gated):
    D, Hk, Hv = shape
    w = small_workload(B=3, S=1, Hk=Hk, Hv=Hv, D=D, act=act, seed=100 + D + Hv, s0_std=0.3)
    inp = make_inputs(w)
    y, st = run_decode(inp, gated=gated)
    yr, sr = oracle_ref(inp, gated=gated)
    assert rel_err(y, yr) <= DECODE_TOL
    assert rel_err(st, sr) <= DECODE_TOL


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_decode_gates_in_activation_dtype(act):
    w = small_workload(B=4, S=1, Hk=2, Hv=4, D=128, act=act, seed=7)
    inp = make_inputs(w, gate_dtype=w.act_dtype)
    y, st = run_decode(inp)
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= DECODE_TOL and rel_err(st, sr) <= DECODE_TOL


def test_decode_head_major_flag_is_a_shape_change_at_one_token():
    w = small_workload(B=5, S=1, Hk=2, Hv=4, D=64, act="bf16", seed=8)
    inp = make_inputs(w)
    y0, s0 = run_decode(inp, head_major=False)
    hm = dict(inp)
    for name in ("q", "k", "v", "z"):
        hm[name] = inp[name].transpose(1, 2).contiguous()
    for name in ("log_decay", "beta"):
        hm[name] = inp[name].transpose(1, 2).contiguous()
    y1, s1 = run_decode(hm, head_major=True)
    assert torch.equal(y1.transpose(1, 2), y0) and torch.equal(s1, s0)


def test_decode_fixed_point_alpha_one_beta_zero_is_exact():
    w = small_workload(B=2, S=1, Hk=1, Hv=2, D=128, seed=9)
    inp = make_inputs(w)
    inp["log_decay"] = torch.zeros_like(inp["log_decay"])
    inp["beta"] = torch.zeros_like(inp["beta"])
    _, st = run_decode(inp)
    assert torch.equal(st.cpu(), inp["s0"])


def test_decode_zero_key_and_query_stay_finite():
    w = small_workload(B=1, S=1, Hk=1, Hv=2, D=64, seed=10)
    inp = make_inputs(w)
    inp["k"] = torch.zeros_like(inp["k"])
    inp["q"] = torch.zeros_like(inp["q"])
    y, st = run_decode(inp)
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= DECODE_TOL and rel_err(st, sr) <= DECODE_TOL


def test_decode_empty_batch_is_a_noop():
    w = small_workload(B=0, S=1, Hk=1, Hv=2, D=16)
    inp = make_inputs(w)
    y, st = run_decode(inp)
    assert y.numel() == 0 and st.numel() == 0


def test_decode_rejects_on_device_without_touching_buffers():
    w = small_workload(B=2, S=1, Hk=1, Hv=2, D=32)
    d = to_dev(make_inputs(w))
    st = d["s0"].clone()
    with pytest.raises(gdn.GdnError, match="z and gn"):
        gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st, z=d["z"])
    torch.cuda.synchronize()
    assert torch.equal(st, d["s0"])
