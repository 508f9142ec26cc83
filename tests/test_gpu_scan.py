"""GPU parity of gdn_scan against the fp64 oracle (through the C ABI).

Tolerance: max |gpu - oracle| / (1 + |oracle|) <= 2e-3 on y and on the final state.  The
full-size prefill and long-context workloads are compared in full (every head, every token)
with the oracle running on all host cores.
"""
from __future__ import annotations

import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import (LONG_B2, PREFILL_B4, TINY,
                                                             make_inputs)
from gdn_testutil import (DECODE_TOL, SCAN_TOL, guard_intact, guarded, oracle_ref,
                          record_margin, rel_err, small_workload, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


def run_scan(inp, *, gated=True, head_major=False, s0="inp"):
    d = to_dev(inp)
    s0v = d["s0"] if s0 == "inp" else s0
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=s0v,
                         z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                         head_major=head_major)
    torch.cuda.synchronize()
    return y, st


def test_tiny_workload():
    inp = make_inputs(TINY)
    y, st = run_scan(inp)
    yr, sr = oracle_ref(inp)
    assert y.shape == (1, 8, 2, 16) and st.shape == (1, 2, 16, 16)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
    # far inside the bar: the tensor-core products split every f32 operand into bf16 hi + lo
    # parts (about 2^-16 relative error per product), so a few 1e-5 at this size
    assert rel_err(y, yr) <= 1e-4


@pytest.mark.parametrize("kernel", ["chunked", "block16"])
@pytest.mark.parametrize("gated", [True, False], ids=["gated", "raw_o"])
@pytest.mark.parametrize("w", [PREFILL_B4, LONG_B2], ids=lambda w: w.name)
def test_full_size_scan_matches_oracle(w, gated, kernel):
    # raw o (no gated norm) as well: rmsnorm would hide a wrong scale on o; both the chunked
    # kernel and the 16-token block kernel
    inp = make_inputs(w)
    d = to_dev(inp)
    y, ywhole = guarded(tuple(d["v"].shape))
    st, swhole = guarded((w.B, w.Hv, w.Dv, w.Dk))
    gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st, y, s0=d["s0"],
                 z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                 head_major=w.head_major, block16=kernel == "block16", chunked=kernel == "chunked")
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    del d
    yr, sr = oracle_ref(inp, gated=gated, head_major=w.head_major)
    ey, es = rel_err(y, yr), rel_err(st, sr)
    name = ("gdn_scan chunked WY (GDN_FLAG_SCAN_CHUNKED)" if kernel == "chunked"
            else "gdn_scan 16-token block (GDN_FLAG_SCAN_BLOCK16)")
    record_margin(w.name, name, "gated y" if gated else "raw o", ey, es, SCAN_TOL)
    assert ey <= SCAN_TOL
    assert es <= SCAN_TOL
    assert guard_intact(ywhole, y.numel()) and guard_intact(swhole, st.numel())


# sequence lengths around the 32-token staging chunk, head dims, GQA ratios, layouts
EDGE = [
    # B, S, Hk, Hv, D, act, head_major
    (1, 1, 1, 1, 16, "f32", False),
    (2, 7, 1, 2, 16, "bf16", True),
    (1, 31, 2, 2, 32, "f16", False),
    (1, 32, 2, 4, 32, "bf16", True),
    (2, 33, 1, 4, 64, "f32", False),
    (1, 65, 2, 4, 64, "bf16", True),
    (1, 100, 1, 2, 128, "f16", False),
    (3, 64, 2, 4, 128, "bf16", True),
    (1, 37, 1, 1, 128, "f32", False),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "_".join(map(str, c)))
@pytest.mark.parametrize("gated", [True, False])
def test_scan_edge_shapes(case, gated):
    B, S, Hk, Hv, D, act, hm = case
    w = small_workload(B=B, S=S, Hk=Hk, Hv=Hv, D=D, act=act, head_major=hm,
                       seed=200 + S + D, s0_std=0.2)
    inp = make_inputs(w)
    y, st = run_scan(inp, gated=gated, head_major=hm)
    yr, sr = oracle_ref(inp, gated=gated, head_major=hm)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL


@pytest.mark.parametrize("heads", [1, 8, 40, 160])
def test_scan_row_split_variants(heads):
    # B*Hv decides how many CTAs share a head (one CTA per head, or a split head with the
    # separate gated-norm kernel); every variant must agree with the oracle.
    Hv = 8 if heads >= 8 else heads
    B = heads // Hv
    w = small_workload(B=B, S=40, Hk=2 if Hv >= 2 else 1, Hv=Hv, D=128, act="bf16",
                       seed=300 + heads, s0_std=0.02, ldr=(-4.0, 0.0))
    inp = make_inputs(w)
    y, st = run_scan(inp)
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
    y, st = run_scan(inp, gated=False)
    yr, sr = oracle_ref(inp, gated=False)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL


def test_scan_zero_initial_state_null_and_buffer_agree():
    w = small_workload(B=2, S=50, Hk=2, Hv=4, D=128, act="bf16", s0_std=None, seed=11)
    inp = make_inputs(w)
    y0, s0 = run_scan(inp, s0=None)
    y1, s1 = run_scan(inp, s0=torch.zeros(2, 4, 128, 128, device="cuda"))
    assert torch.equal(y0, y1) and torch.equal(s0, s1)
    yr, sr = oracle_ref(inp, s0=None)
    assert rel_err(y0, yr) <= SCAN_TOL and rel_err(s0, sr) <= SCAN_TOL


def test_scan_in_place_resume_and_split_equal_single_scan():
    w = small_workload(B=2, S=90, Hk=1, Hv=4, D=64, act="bf16", seed=12)
    d = to_dev(make_inputs(w))
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                         z=d["z"], gn=d["gn"])
    state = d["s0"].clone()
    parts = []
    for a, b in ((0, 33), (33, 34), (34, 90)):
        sl = {k: d[k][:, a:b].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
        yp, _ = gdn.gdn_scan(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"], state,
                             s0=state, z=sl["z"], gn=d["gn"])
        parts.append(yp)
    torch.cuda.synchronize()
    # the same recurrence, but the kernel's deferred decay restarts at each call, so the two
    # evaluations agree to f32 rounding rather than bit for bit
    ys = torch.cat(parts, 1)
    assert float(((ys - y).abs() / (1 + y.abs())).max()) <= DECODE_TOL
    assert float(((state - st).abs() / (1 + st.abs())).max()) <= DECODE_TOL


def test_decode_steps_equal_scan():
    w = small_workload(B=2, S=12, Hk=2, Hv=4, D=128, act="bf16", seed=13, s0_std=0.02)
    d = to_dev(make_inputs(w))
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                         z=d["z"], gn=d["gn"])
    state = d["s0"].clone()
    ys = []
    for t in range(12):
        sl = {k: d[k][:, t:t + 1].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
        ys.append(gdn.gdn_decode_step(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"],
                                      state, z=sl["z"], gn=d["gn"]))
    torch.cuda.synchronize()
    yd = torch.cat(ys, 1)
    err_y = float(((yd - y).abs() / (1 + y.abs())).max())
    err_s = float(((state - st).abs() / (1 + st.abs())).max())
    assert err_y <= DECODE_TOL and err_s <= DECODE_TOL


def test_scan_head_major_equals_seq_major():
    w = small_workload(B=2, S=45, Hk=2, Hv=4, D=64, act="f16", seed=14)
    inp = make_inputs(w)
    y0, s0 = run_scan(inp)
    hm = dict(inp)
    for name in ("q", "k", "v", "z", "log_decay", "beta"):
        hm[name] = inp[name].transpose(1, 2).contiguous()
    y1, s1 = run_scan(hm, head_major=True)
    assert torch.equal(y1.transpose(1, 2), y0) and torch.equal(s1, s0)


def test_scan_gqa_equals_explicit_repeat():
    w = small_workload(B=1, S=20, Hk=2, Hv=8, D=32, act="bf16", seed=15)
    inp = make_inputs(w)
    y0, s0 = run_scan(inp)
    rep = dict(inp)
    rep["q"] = inp["q"].repeat_interleave(4, dim=2)
    rep["k"] = inp["k"].repeat_interleave(4, dim=2)
    y1, s1 = run_scan(rep)
    assert torch.equal(y0, y1) and torch.equal(s0, s1)


def test_scan_empty_sequence_copies_state():
    w = small_workload(B=2, S=0, Hk=1, Hv=2, D=32, seed=16)
    inp = make_inputs(w)
    y, st = run_scan(inp)
    assert y.numel() == 0 and torch.equal(st.cpu(), inp["s0"])
    _, st0 = run_scan(inp, s0=None)
    assert torch.count_nonzero(st0) == 0


def test_scan_gates_in_activation_dtype():
    w = small_workload(B=1, S=70, Hk=1, Hv=2, D=128, act="bf16", seed=17)
    inp = make_inputs(w, gate_dtype=torch.bfloat16)
    y, st = run_scan(inp)
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
