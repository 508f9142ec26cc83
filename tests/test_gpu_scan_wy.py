"""GPU parity of the chunked (WY-form, tcgen05) scan kernel against the fp64 oracle.

The kernel applies to bf16 and f16 activations with Dk = Dv = 128; these tests select it with
GDN_FLAG_SCAN_CHUNKED (the default picks it or the block kernel by shape, checked last).  It
writes the page's per-token recurrence (logicaffeine codegen_cuda::gdn, module description)
exactly over chunks of 64 tokens: the chunk's corrections D = U - W S^T with U, W from the
unit-triangular inverse T = (I + A)^-1, the outputs from the chunk-start memory plus the
intra-chunk term, and the chunk-end memory.  The cases cross chunk boundaries (1, 63, 64, 65,
127, 128, 129 tokens and longer), both activation types, both layouts, grouped heads, gated and
raw outputs, zero, given and in-place initial memory, slow decay and decay fast enough that a
chunk's cumulative product underflows, gates in the activation type, and compare with the
16-token block kernel (GDN_FLAG_SCAN_BLOCK16).  Tolerance: 2e-3 relative to 1 + |oracle|.
"""
from __future__ import annotations

import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import make_inputs
from gdn_testutil import SCAN_TOL, oracle_ref, rel_err, small_workload, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


def run(d, *, gated=True, head_major=False, s0="inp", block16=False, auto=False):
    s0v = d["s0"] if s0 == "inp" else s0
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=s0v,
                         z=d["z"] if gated else None, gn=d["gn"] if gated else None,
                         head_major=head_major, block16=block16,
                         chunked=not block16 and not auto)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    return y, st


CASES = [
    # B, S, Hk, Hv, act, head_major, log_decay range
    (1, 1, 1, 1, "bf16", False, (-3.0, 0.0)),
    (1, 63, 1, 2, "bf16", False, (-3.0, 0.0)),
    (1, 64, 1, 1, "f16", False, (-3.0, 0.0)),
    (1, 65, 2, 2, "bf16", True, (-3.0, 0.0)),
    (2, 127, 1, 2, "f16", False, (-4.0, 0.0)),
    (1, 128, 1, 4, "bf16", False, (-8.0, -3.0)),
    (1, 129, 2, 4, "f16", True, (-8.0, -3.0)),
    (3, 200, 1, 3, "bf16", False, (-4.0, 0.0)),
    (1, 777, 1, 2, "f16", False, (-4.0, 0.0)),
    (1, 300, 1, 1, "bf16", False, (2.0, 3.0)),      # log_decay down to -20 per token
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c)))
@pytest.mark.parametrize("gated", [True, False], ids=["gated", "raw_o"])
def test_chunked_scan_matches_oracle(case, gated):
    B, S, Hk, Hv, act, hm, ldr = case
    w = small_workload(B=B, S=S, Hk=Hk, Hv=Hv, D=128, act=act, head_major=hm,
                       seed=500 + S + Hv, s0_std=0.05, ldr=ldr)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = run(d, gated=gated, head_major=hm)
    yr, sr = oracle_ref(inp, gated=gated, head_major=hm)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
    # far inside the bar: every f32 operand enters as hi + lo parts
    assert rel_err(st, sr) <= 1e-4


def test_chunked_scan_agrees_with_block_kernel():
    w = small_workload(B=2, S=333, Hk=2, Hv=4, D=128, act="bf16", seed=601, s0_std=0.05,
                       ldr=(-4.0, 0.0))
    d = to_dev(make_inputs(w))
    y0, s0 = run(d)
    y1, s1 = run(d, block16=True)
    assert float(((y0 - y1).abs() / (1 + y1.abs())).max()) <= SCAN_TOL
    assert float(((s0 - s1).abs() / (1 + s1.abs())).max()) <= SCAN_TOL


def test_chunked_scan_zero_state_null_buffer_and_in_place_resume():
    w = small_workload(B=1, S=150, Hk=1, Hv=2, D=128, act="bf16", seed=602, s0_std=None)
    inp = make_inputs(w)
    d = to_dev(inp)
    y0, s0 = run(d, s0=None)
    y1, s1 = run(d, s0=torch.zeros(1, 2, 128, 128, device="cuda"))
    assert torch.equal(y0, y1) and torch.equal(s0, s1)
    yr, sr = oracle_ref(inp, s0=None)
    assert rel_err(y0, yr) <= SCAN_TOL and rel_err(s0, sr) <= SCAN_TOL
    # resume in place over two calls (50 + 100 tokens): state is s0 of the second call
    state = torch.zeros(1, 2, 128, 128, device="cuda")
    parts = []
    for a, b in ((0, 50), (50, 150)):
        sl = {k: d[k][:, a:b].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
        yp, _ = gdn.gdn_scan(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"], state,
                             s0=state, z=sl["z"], gn=d["gn"], chunked=True)
        parts.append(yp)
    torch.cuda.synchronize()
    assert rel_err(torch.cat(parts, 1), yr) <= SCAN_TOL and rel_err(state, sr) <= SCAN_TOL


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_chunked_scan_gates_in_activation_dtype(act):
    w = small_workload(B=1, S=140, Hk=1, Hv=2, D=128, act=act, seed=603, s0_std=0.05)
    dt = torch.bfloat16 if act == "bf16" else torch.float16
    inp = make_inputs(w, gate_dtype=dt)
    y, st = run(to_dev(inp))
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL


def test_chunked_scan_many_heads_and_zero_keys():
    # more heads than SMs (several CTA waves), and zero k / q rows (k^ = 0: a pure decay step)
    w = small_workload(B=5, S=70, Hk=8, Hv=40, D=128, act="bf16", seed=604, s0_std=0.05)
    inp = make_inputs(w)
    inp["k"][:, 10] = 0
    inp["q"][:, 11] = 0
    y, st = run(to_dev(inp))
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL


@pytest.mark.parametrize("act,B,Hv,want", [
    ("f16", 1, 2, "chunked"),          # f16: the chunked kernel at every head count
    ("bf16", 1, 2, "block16"),         # bf16, few heads: the block kernel splits each over CTAs
    ("bf16", 4, 32, "chunked"),        # bf16, 128 heads: the block kernel would run one per CTA
    ("bf16", 4, 80, "chunked"),        # bf16, more heads than SMs: the block kernel would stack
])
def test_default_kernel_choice(act, B, Hv, want):
    # the default runs one of the two kernels bit for bit (which one depends on the head count
    # against this device's SMs: 320 heads exceed any GB300's)
    w = small_workload(B=B, S=40, Hk=Hv // 2 if Hv > 1 else 1, Hv=Hv, D=128, act=act, seed=605,
                       s0_std=0.05)
    d = to_dev(make_inputs(w))
    y0, s0 = run(d, auto=True)
    y1, s1 = run(d, block16=want == "block16")
    assert torch.equal(y0, y1) and torch.equal(s0, s1)
