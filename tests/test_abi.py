"""The C ABI without a GPU: the library loads, exports what include/gdn.h declares, the
ctypes mirror matches the C struct layout, and every rejection happens on the host before
any CUDA call (no compute is launched in this file)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest
import torch

import linear_attention_recurrence_gdn_gb300 as gdn
from linear_attention_recurrence_gdn_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build_library()
    return gdn.library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(gdn.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.LIBRARY], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted({m for m in re.findall(r"\bT (gdn_\w+)", out)})
    assert exported == declared_functions()


def test_struct_layout_matches_header(tmp_path):
    fields = [f[0] for f in gdn.GdnParams._fields_]
    prog = ["#include <stddef.h>", "#include <stdio.h>", '#include "gdn.h"', "int main(void){",
            'printf("%zu\\n", sizeof(gdn_params));']
    prog += [f'printf("%zu\\n", offsetof(gdn_params, {f}));' for f in fields]
    prog += ["return 0;}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                   check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(gdn.GdnParams)
    for f, off in zip(fields, vals[1:]):
        assert getattr(gdn.GdnParams, f).offset == off, f


def test_version_and_status_strings(lib):
    assert gdn.gdn_version() == 1
    codes = [0, -1, -2, -3, -4, -5, -6, -7, -8, -9]
    texts = [gdn.gdn_status_string(c) for c in codes]
    assert len(set(texts)) == len(codes)
    assert gdn.gdn_status_string(12345) == "unknown status"
    assert gdn.gdn_last_error() == ""


# --------------------------------------------------------------- host-side validation

BASE = 1 << 40          # fake, 4 KiB-aligned device addresses: never dereferenced here
GAP = 1 << 32


def fake_params(**kw):
    """A launchable parameter set on fake pointers (B, S, Hk, Hv, D = 2, 3, 2, 4, 64)."""
    p = dict(B=2, S=3, Hk=2, Hv=4, Dk=64, Dv=64, head_major=0, act_dtype=gdn.GDN_BF16,
             gate_dtype=gdn.GDN_F32, flags=0, qk_eps=1e-6, norm_eps=1e-6)
    names = ["q", "k", "v", "log_decay", "beta", "z", "gn", "s0", "state", "y"]
    for i, n in enumerate(names):
        p[n] = BASE + i * GAP
    p.update(kw)
    return gdn.GdnParams(**p)


def reject(lib, prm, is_decode):
    r = lib.gdn_reject_reason(ctypes.byref(prm), is_decode)
    return None if r is None else r.decode()


def call(lib, prm, is_decode):
    fn = lib.gdn_decode_step if is_decode else lib.gdn_scan
    return fn(ctypes.byref(prm), None)


def test_valid_params_have_no_reject_reason(lib):
    assert reject(lib, fake_params(), 0) is None
    assert reject(lib, fake_params(S=1), 1) is None
    assert reject(lib, fake_params(S=1, head_major=1), 1) is None
    assert reject(lib, fake_params(z=None, gn=None), 0) is None          # raw o mode
    assert reject(lib, fake_params(s0=None), 0) is None                 # zeros
    st = BASE + 8 * GAP
    assert reject(lib, fake_params(s0=st, state=st), 0) is None         # in-place resume
    assert reject(lib, fake_params(gate_dtype=gdn.GDN_BF16), 0) is None
    assert reject(lib, fake_params(S=1, flags=gdn.GDN_FLAG_HOST_IO), 1) is None
    assert reject(lib, fake_params(flags=gdn.GDN_FLAG_SCAN_TMEM), 0) is None
    assert reject(lib, fake_params(flags=gdn.GDN_FLAG_SCAN_BLOCK16), 0) is None
    assert reject(lib, fake_params(flags=gdn.GDN_FLAG_SCAN_CHUNKED), 0) is None
    # empty sequence: empty tensors may come as NULL pointers, nothing is read or written
    assert reject(lib, fake_params(S=0, y=None, q=None, k=None, v=None, z=None, log_decay=None,
                                   beta=None), 0) is None
    for d in (16, 32, 128, 256):
        assert reject(lib, fake_params(Dk=d, Dv=d), 0) is None
    # separate key and value head dims
    for dk, dv in ((64, 128), (128, 32), (16, 64), (256, 128), (128, 256), (256, 48)):
        assert reject(lib, fake_params(Dk=dk, Dv=dv), 0) is None
        assert reject(lib, fake_params(Dk=dk, Dv=dv, S=1), 1) is None
    # any other dims whose memory fits the general kernel
    for dk, dv in ((40, 40), (64, 72), (144, 64), (1, 1), (100, 72), (232, 232), (255, 9),
                   (236, 236)):
        assert reject(lib, fake_params(Dk=dk, Dv=dv), 0) is None
        assert reject(lib, fake_params(Dk=dk, Dv=dv, S=1), 1) is None


REJECTIONS = [
    # (overrides, is_decode, status, reason fragment)
    (dict(Hv=3), 0, gdn.GDN_ERR_BAD_SHAPE, "multiple of Hk"),
    (dict(Hk=0), 0, gdn.GDN_ERR_BAD_SHAPE, "Hk and Hv"),
    (dict(B=-1), 0, gdn.GDN_ERR_BAD_SHAPE, "B and S"),
    (dict(S=-2), 0, gdn.GDN_ERR_BAD_SHAPE, "B and S"),
    (dict(S=3), 1, gdn.GDN_ERR_BAD_SHAPE, "S == 1"),
    (dict(S=0), 1, gdn.GDN_ERR_BAD_SHAPE, "S == 1"),
    (dict(Dk=240, Dv=256), 0, gdn.GDN_ERR_UNSUPPORTED_DIM, "226 KB"),   # general: 241 KB
    (dict(Dk=256, Dv=512), 0, gdn.GDN_ERR_UNSUPPORTED_DIM, "at most 256"),
    (dict(Dk=300, Dv=16), 0, gdn.GDN_ERR_UNSUPPORTED_DIM, "at most 256"),
    (dict(Dk=250, Dv=250, S=1), 1, gdn.GDN_ERR_UNSUPPORTED_DIM, "226 KB"),
    (dict(Dk=239, Dv=239), 0, gdn.GDN_ERR_UNSUPPORTED_DIM, "226 KB"),   # rows padded to 244
    (dict(act_dtype=7), 0, gdn.GDN_ERR_BAD_DTYPE, "act_dtype"),
    (dict(act_dtype=gdn.GDN_BF16, gate_dtype=gdn.GDN_F16), 0, gdn.GDN_ERR_BAD_DTYPE, "gate_dtype"),
    (dict(qk_eps=-1.0), 0, gdn.GDN_ERR_BAD_ARG, "eps"),
    (dict(norm_eps=float("nan")), 0, gdn.GDN_ERR_BAD_ARG, "eps"),
    (dict(norm_eps=float("inf")), 0, gdn.GDN_ERR_BAD_ARG, "eps"),
    (dict(head_major=2), 0, gdn.GDN_ERR_BAD_ARG, "head_major"),
    (dict(flags=16), 0, gdn.GDN_ERR_BAD_ARG, "unknown flags"),
    (dict(S=1, flags=32), 1, gdn.GDN_ERR_BAD_ARG, "unknown flags"),
    (dict(S=1, flags=gdn.GDN_FLAG_SCAN_CHUNKED), 1, gdn.GDN_ERR_BAD_ARG, "gdn_scan only"),
    (dict(flags=gdn.GDN_FLAG_SCAN_CHUNKED | gdn.GDN_FLAG_SCAN_BLOCK16), 0, gdn.GDN_ERR_BAD_ARG,
     "at most one"),
    (dict(flags=gdn.GDN_FLAG_SCAN_TMEM | gdn.GDN_FLAG_SCAN_BLOCK16), 0, gdn.GDN_ERR_BAD_ARG,
     "at most one"),
    (dict(S=1, flags=gdn.GDN_FLAG_SCAN_BLOCK16), 1, gdn.GDN_ERR_BAD_ARG, "gdn_scan only"),
    (dict(S=1, flags=gdn.GDN_FLAG_SCAN_TMEM), 1, gdn.GDN_ERR_BAD_ARG, "gdn_scan only"),
    (dict(flags=gdn.GDN_FLAG_HOST_IO), 0, gdn.GDN_ERR_BAD_ARG, "gdn_decode_step only"),
    (dict(B=1 << 20, S=1 << 20), 0, gdn.GDN_ERR_BAD_ARG, "too large"),
    (dict(state=None), 0, gdn.GDN_ERR_NULL_PTR, "state and y"),
    (dict(S=1, y=None), 1, gdn.GDN_ERR_NULL_PTR, "state and y"),
    (dict(q=None), 0, gdn.GDN_ERR_NULL_PTR, "required"),
    (dict(beta=None), 0, gdn.GDN_ERR_NULL_PTR, "required"),
    (dict(z=None), 0, gdn.GDN_ERR_NULL_PTR, "z and gn"),
    (dict(gn=None), 0, gdn.GDN_ERR_NULL_PTR, "z and gn"),
    (dict(q=BASE + 8), 0, gdn.GDN_ERR_MISALIGNED, "16-byte"),
    (dict(S=1, state=BASE + 8 * GAP + 4), 1, gdn.GDN_ERR_MISALIGNED, "16-byte"),
    (dict(log_decay=BASE + 3 * GAP + 2), 0, gdn.GDN_ERR_MISALIGNED, "element size"),
    (dict(y=BASE), 0, gdn.GDN_ERR_ALIASING, "y overlaps"),                     # y == q
    (dict(S=1, y=BASE + 8 * GAP + 1024), 1, gdn.GDN_ERR_ALIASING, "y overlaps"),    # inside state
    (dict(state=BASE + 2 * GAP + 1024), 0, gdn.GDN_ERR_ALIASING, "state overlaps"),
    (dict(s0=BASE + 8 * GAP + 256), 0, gdn.GDN_ERR_ALIASING, "partially overlaps s0"),
]


@pytest.mark.parametrize("case", REJECTIONS, ids=lambda c: c[3] + str(sorted(c[0])))
def test_rejections_return_before_any_launch(lib, case):
    kw, is_decode, status, fragment = case
    prm = fake_params(**kw)
    reason = reject(lib, prm, is_decode)
    assert reason is not None and fragment in reason, reason
    assert call(lib, prm, is_decode) == status


def test_split_scan_rejections_return_before_any_launch(lib):
    # fake_params: B 2, S 3, Hk 2, Hv 4, D 64 -> 2 segments of 2 and 1 tokens; workspace of
    # M, N for one segment and starts for two: (8*64*64 * (1 + 1 + 2)) floats
    prm = fake_params()
    need = lib.gdn_scan_split_workspace(ctypes.byref(prm), 2)
    assert need == 4 * 8 * 64 * 64 * 4
    assert lib.gdn_scan_split_workspace(ctypes.byref(prm), 1) == 0
    assert lib.gdn_scan_split_workspace(ctypes.byref(fake_params(Hv=3)), 2) == 0   # rejected p
    ws = BASE + 16 * GAP
    cases = [
        (dict(), 0, ws, need, gdn.GDN_ERR_BAD_ARG, "segments"),
        (dict(flags=gdn.GDN_FLAG_SCAN_TMEM), 2, ws, need, gdn.GDN_ERR_BAD_ARG, "gdn_scan only"),
        (dict(), 2, None, need, gdn.GDN_ERR_NULL_PTR, "workspace is required"),
        (dict(), 2, ws + 8, need, gdn.GDN_ERR_MISALIGNED, "16-byte"),
        (dict(), 2, ws, need - 16, gdn.GDN_ERR_BAD_ARG, "too small"),
        (dict(), 2, BASE + 9 * GAP - 64, need, gdn.GDN_ERR_ALIASING, "overlaps"),   # into y
        (dict(Hv=3), 2, ws, need, gdn.GDN_ERR_BAD_SHAPE, ""),        # gdn_scan's own checks
    ]
    for kw, nseg, w, nbytes, status, fragment in cases:
        p = fake_params(**kw)
        assert lib.gdn_scan_split(ctypes.byref(p), nseg, w, nbytes, None) == status, kw
        if fragment:
            assert fragment in lib.gdn_last_error().decode()


def test_null_params_pointer(lib):
    assert lib.gdn_scan(None, None) == gdn.GDN_ERR_NULL_PTR
    assert lib.gdn_decode_step(None, None) == gdn.GDN_ERR_NULL_PTR
    assert lib.gdn_reject_reason(None, 0).decode() == "params pointer is NULL"


def test_empty_batch_is_a_noop_without_cuda(lib):
    # B == 0 returns OK before touching CUDA, even with NULL data pointers
    prm = fake_params(B=0, q=None, k=None, v=None, state=None, y=None)
    assert call(lib, prm, 0) == gdn.GDN_OK
    assert call(lib, fake_params(B=0, S=1), 1) == gdn.GDN_OK


def test_decode_ignores_s0_overlap(lib):
    # decode never reads s0, so an s0 that overlaps state is not an error there
    st = BASE + 8 * GAP
    assert reject(lib, fake_params(S=1, s0=st + 256, state=st), 1) is None


# ----------------------------------------------------------- binding-side marshalling

def test_binding_rejects_cpu_tensors_and_noncontiguous():
    q = torch.zeros(1, 1, 1, 16)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_decode_step(q, q, q, torch.zeros(1, 1, 1), torch.zeros(1, 1, 1),
                            torch.zeros(1, 1, 16, 16))
    t = torch.zeros(1, 1, 1, 32)[..., ::2]
    with pytest.raises(gdn.GdnError, match="contiguous"):
        gdn.make_params(t, t, t, torch.zeros(1, 2, 1), torch.zeros(1, 2, 1),
                        torch.zeros(1, 1, 16, 16), torch.zeros(1, 1, 1, 16))


def test_binding_host_io_refuses_unpinned_host_tensors():
    # GDN_FLAG_HOST_IO operands must be device-addressable: CUDA tensors or pinned host
    # memory; ordinary (pageable) CPU tensors are refused before any CUDA call
    q = torch.zeros(1, 1, 1, 16)
    with pytest.raises(gdn.GdnError, match="pinned"):
        gdn.gdn_decode_step(q, q, q, torch.zeros(1, 1, 1), torch.zeros(1, 1, 1),
                            torch.zeros(1, 1, 16, 16), host_io=True)


def test_binding_split_scan_refuses_cpu_tensors():
    # no CPU path: the sequence-split scan, like the scan, takes CUDA tensors only
    q = torch.zeros(1, 4, 1, 16)
    g = torch.zeros(1, 4, 1)
    with pytest.raises(gdn.GdnError, match="CUDA"):
        gdn.gdn_scan_split(q, q, q, g, g, segments=2)


def test_binding_shape_and_dtype_checks():
    B, S, Hk, Hv, D = 1, 2, 1, 2, 16
    q = torch.zeros(B, S, Hk, D, dtype=torch.bfloat16)
    v = torch.zeros(B, S, Hv, D, dtype=torch.bfloat16)
    g = torch.zeros(B, S, Hv)
    st = torch.zeros(B, Hv, D, D)
    y = torch.zeros(B, S, Hv, D)
    prm = gdn.make_params(q, q, v, g, g, st, y, head_major=False)
    assert (prm.B, prm.S, prm.Hk, prm.Hv, prm.Dk, prm.Dv) == (1, 2, 1, 2, 16, 16)
    assert prm.act_dtype == gdn.GDN_BF16 and prm.gate_dtype == gdn.GDN_F32
    with pytest.raises(gdn.GdnError, match="shape"):
        gdn.make_params(q, q, v, g, g, st, torch.zeros(B, S, Hv, D + 1))
    with pytest.raises(gdn.GdnError, match="dtype"):
        gdn.make_params(q, q, v.float(), g, g, st, y)
    with pytest.raises(gdn.GdnError, match="float32"):
        gdn.make_params(q, q, v, g, g, st.double(), y)
    hm = gdn.make_params(q.transpose(1, 2).contiguous(), q.transpose(1, 2).contiguous(),
                         v.transpose(1, 2).contiguous(), g.transpose(1, 2).contiguous(),
                         g.transpose(1, 2).contiguous(), st, y.transpose(1, 2).contiguous(),
                         head_major=True)
    assert (hm.B, hm.S, hm.Hk, hm.Hv) == (1, 2, 1, 2) and hm.head_major == 1


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        gdn.library(str(tmp_path / "libgdn.so"))


def test_selftest_wait_timeout_rejects_bad_limits_without_a_gpu(lib):
    # argument checks run before any CUDA call
    for bad in (0.0, -1.0, 2000.5, float("nan")):
        assert lib.gdn_selftest_wait_timeout(None, bad) == -7   # GDN_ERR_BAD_ARG
