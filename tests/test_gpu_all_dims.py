"""Every supported head-dim pair and activation type through both entry points, on a tiny
case against the fp64 oracle: Dk and Dv each 16, 32, ..., 128 or 256, f32 / bf16 / f16.

Each (type, Dk, Dv) has its own kernel instantiation and its own launch choice (rows per CTA,
pipeline stages, shared-memory size); this sweep shows that every one launches on this device
and computes the recurrence.  Three tokens cross no chunk boundary, so the deep cases live in
the other files; here the point is coverage of the dispatch.  Tolerances as everywhere:
decode 1e-4, scan 2e-3 (relative to 1 + |oracle|).
"""
from __future__ import annotations

import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild
from linear_attention_recurrence_gdn_gb300.workloads import make_inputs
from gdn_testutil import DECODE_TOL, SCAN_TOL, oracle_ref, rel_err, small_workload, to_dev

pytestmark = pytest.mark.gpu

DIMS = [16, 32, 48, 64, 80, 96, 112, 128, 256]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build_library()
    gdn.library()


@pytest.mark.parametrize("act", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("dk", DIMS)
@pytest.mark.parametrize("dv", DIMS)
def test_every_head_dim_pair_scan_and_decode(act, dk, dv):
    w = small_workload(B=1, S=3, Hk=1, Hv=2, Dk=dk, Dv=dv, act=act, seed=900 + dk + 7 * dv,
                       s0_std=0.05)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], s0=d["s0"],
                         z=d["z"], gn=d["gn"])
    state = d["s0"].clone()
    sl = {k: d[k][:, :1].contiguous() for k in ("q", "k", "v", "z", "log_decay", "beta")}
    y1 = gdn.gdn_decode_step(sl["q"], sl["k"], sl["v"], sl["log_decay"], sl["beta"], state,
                             z=sl["z"], gn=d["gn"])
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    yr, sr = oracle_ref(inp)
    assert rel_err(y, yr) <= SCAN_TOL and rel_err(st, sr) <= SCAN_TOL
    one = {k: (v[:, :1].contiguous() if v is not None and v.dim() >= 3 and k != "s0" else v)
           for k, v in inp.items()}
    yr1, sr1 = oracle_ref(one)
    assert rel_err(y1, yr1) <= DECODE_TOL and rel_err(state, sr1) <= DECODE_TOL
