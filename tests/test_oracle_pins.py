"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

The oracle (``oracle/gdn_oracle.c``) is checked here against things other than itself:

* a 50-digit decimal brute force of the closed-form update (``oracle/closed_form_decimal``)
  and golden fixtures written by it;
* fixed points and closed forms of the recurrence of the logicaffeine
  ``codegen_cuda::gdn`` page (module description): alpha=1/beta=0 leaves S unchanged,
  beta=0 is pure decay, an empty memory after one token holds beta v k^T, the delta rule
  retrieves v at beta=1;
* the single-pass identity of that page's "The fusion" section against the literal
  three-pass evaluation;
* exact invariances (scaling by a power of two, permutations of key dim, value dim, value
  heads within a group and key groups -- the "function-preserving" permutations of
  modelopt's gated_delta_net page), compositions (split scan, decode steps, head_major,
  GQA against explicit repetition) and the gated norm against torch's rms_norm/silu.
"""
from __future__ import annotations

import glob
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import closed_form_decimal
from linear_attention_recurrence_gdn_gb300.workloads import TINY, make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def small(B=1, S=3, Hk=1, Hv=1, D=4, *, head_major=False, s0_std=0.1, seed=7,
          ldr=(-3.0, 0.0), act="f32", Dk=None, Dv=None):
    w = TINY.replace(name="small", B=B, S=S, Hk=Hk, Hv=Hv, Dk=Dk or D, Dv=Dv or D,
                     head_major=head_major,
                     s0_std=s0_std, seed=seed, log_decay_range=ldr, act=act)
    inp = {k: (None if v is None else v.double()) for k, v in make_inputs(w).items()}
    return w, inp


def orun(inp, *, gated=True, head_major=False, mode="literal", **kw):
    args = dict(z=inp["z"] if gated else None, gn=inp["gn"] if gated else None,
                s0=inp["s0"], head_major=head_major, mode=mode)
    args.update(kw)
    return oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"], **args)


def rel_err(a, ref):
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(a - ref) / (1.0 + np.abs(ref)))) if ref.size else 0.0


def qhat(q):
    """q / sqrt(sum q^2 + eps) / sqrt(Dk) on a float64 array (last axis)."""
    q = np.asarray(q, dtype=np.float64)
    return q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6) / np.sqrt(q.shape[-1])


def khat(k):
    k = np.asarray(k, dtype=np.float64)
    return k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)


# --------------------------------------------------------------------------- decimal pins

DECIMAL_CASES = [
    # B, S, Hk, Hv, D, head_major, gated, s0_std, seed
    (1, 8, 2, 2, 16, False, True, 0.1, 1001),   # the tiny f32 workload's shape
    (2, 3, 1, 2, 4, False, False, 0.1, 21),
    (1, 4, 2, 4, 8, True, True, 0.1, 22),
    (1, 2, 1, 4, 4, False, False, None, 23),
    (1, 5, 2, 4, 4, True, False, 0.3, 24),
]


@pytest.mark.parametrize("case", DECIMAL_CASES, ids=lambda c: "x".join(map(str, c[:5])))
@pytest.mark.parametrize("mode", ["literal", "fused"])
def test_oracle_matches_decimal_closed_form(case, mode):
    B, S, Hk, Hv, D, hm, gated, s0_std, seed = case
    _, inp = small(B, S, Hk, Hv, D, head_major=hm, s0_std=s0_std, seed=seed)
    y, st = orun(inp, gated=gated, head_major=hm, mode=mode)
    yd, sd = closed_form_decimal.run(
        inp["q"].numpy(), inp["k"].numpy(), inp["v"].numpy(), inp["log_decay"].numpy(),
        inp["beta"].numpy(), z=inp["z"].numpy() if gated else None,
        gn=inp["gn"].numpy() if gated else None,
        s0=None if inp["s0"] is None else inp["s0"].numpy(), head_major=hm)
    assert rel_err(y, yd) <= 1e-12
    assert rel_err(st, sd) <= 1e-12


# separate key and value head dims: a transposed index anywhere (state rows vs columns, the
# norm's axis, q / k vs v / z strides) fails these
RECT_CASES = [
    # B, S, Hk, Hv, Dk, Dv, head_major, gated, seed
    (1, 4, 1, 2, 3, 5, False, True, 31),
    (2, 3, 1, 2, 6, 2, True, True, 32),
    (1, 5, 2, 4, 4, 7, False, False, 33),
]


@pytest.mark.parametrize("case", RECT_CASES, ids=lambda c: "x".join(map(str, c[:6])))
@pytest.mark.parametrize("mode", ["literal", "fused"])
def test_oracle_matches_decimal_closed_form_rectangular_heads(case, mode):
    B, S, Hk, Hv, Dk, Dv, hm, gated, seed = case
    _, inp = small(B, S, Hk, Hv, head_major=hm, seed=seed, Dk=Dk, Dv=Dv)
    y, st = orun(inp, gated=gated, head_major=hm, mode=mode)
    assert st.shape == (B, Hv, Dv, Dk)
    yd, sd = closed_form_decimal.run(
        inp["q"].numpy(), inp["k"].numpy(), inp["v"].numpy(), inp["log_decay"].numpy(),
        inp["beta"].numpy(), z=inp["z"].numpy() if gated else None,
        gn=inp["gn"].numpy() if gated else None, s0=inp["s0"].numpy(), head_major=hm)
    assert rel_err(y, yd) <= 1e-12
    assert rel_err(st, sd) <= 1e-12


def test_tiny_workload_itself_against_decimal():
    inp = {k: (None if v is None else v.double()) for k, v in make_inputs(TINY).items()}
    y, st = orun(inp)
    yd, sd = closed_form_decimal.run(
        inp["q"].numpy(), inp["k"].numpy(), inp["v"].numpy(), inp["log_decay"].numpy(),
        inp["beta"].numpy(), z=inp["z"].numpy(), gn=inp["gn"].numpy(), s0=inp["s0"].numpy())
    assert y.shape == (1, 8, 2, 16) and st.shape == (1, 2, 16, 16)
    assert rel_err(y, yd) <= 1e-12 and rel_err(st, sd) <= 1e-12


def _unpack(d):
    return np.array([float.fromhex(h) for h in d["hex"]], dtype=np.float64).reshape(d["shape"])


GOLDEN = sorted(glob.glob(os.path.join(HERE, "golden", "gdn_*.json")))


@pytest.mark.parametrize("path", GOLDEN, ids=lambda p: os.path.basename(p))
@pytest.mark.parametrize("mode", ["literal", "fused"])
def test_golden_fixture(path, mode):
    with open(path) as f:
        g = json.load(f)
    inp = {k: _unpack(v) for k, v in g["inputs"].items()}
    y, st = oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                       z=inp.get("z"), gn=inp.get("gn"), s0=inp.get("s0"),
                       head_major=g["head_major"], qk_eps=g["qk_eps"], norm_eps=g["norm_eps"],
                       mode=mode)
    assert rel_err(y, _unpack(g["expected"]["y"])) <= 1e-12
    assert rel_err(st, _unpack(g["expected"]["state"])) <= 1e-12


def test_golden_fixtures_present():
    assert len(GOLDEN) >= 3


# ---------------------------------------------------------------- fusion identity

@pytest.mark.parametrize("shape", [(2, 5, 2, 4, 32), (1, 7, 1, 2, 64), (1, 3, 4, 4, 128)])
@pytest.mark.parametrize("gated", [False, True])
def test_fused_identity_matches_literal(shape, gated):
    B, S, Hk, Hv, D = shape
    _, inp = small(B, S, Hk, Hv, D, seed=31 + D)
    y1, s1 = orun(inp, gated=gated, mode="literal")
    y2, s2 = orun(inp, gated=gated, mode="fused")
    assert rel_err(y2, y1) <= 1e-12
    assert rel_err(s2, s1) <= 1e-12


# ------------------------------------------------------------ fixed points / closed forms

def test_alpha_one_beta_zero_leaves_memory_unchanged():
    _, inp = small(2, 6, 2, 4, 8, seed=41)
    inp["log_decay"] = torch.zeros_like(inp["log_decay"])
    inp["beta"] = torch.zeros_like(inp["beta"])
    y, st = orun(inp, gated=False)
    assert np.array_equal(st, inp["s0"].numpy())          # exactly unchanged
    # raw o = S0 q^ for every token, with the key head of each value head
    s0 = inp["s0"].numpy()
    qh = qhat(inp["q"].numpy())                            # [B,S,Hk,D]
    qh_v = np.repeat(qh, 2, axis=2)                        # value head hv -> key head hv//2
    expect = np.einsum("bhaj,bthj->btha", s0, qh_v)
    assert rel_err(y, expect) <= 1e-13


def test_pure_decay_closed_form():
    _, inp = small(1, 9, 1, 2, 8, seed=42)
    inp["beta"] = torch.zeros_like(inp["beta"])
    _, st = orun(inp, gated=False)
    total = inp["log_decay"].numpy().sum(axis=1)           # [B,Hv]
    expect = np.exp(total)[:, :, None, None] * inp["s0"].numpy()
    assert rel_err(st, expect) <= 1e-13


def test_empty_memory_one_token():
    _, inp = small(2, 1, 2, 4, 8, s0_std=None, seed=43)
    y, st = orun(inp, gated=False)
    kh = np.repeat(khat(inp["k"].numpy()), 2, axis=2)[:, 0]     # [B,Hv,D]
    qh = np.repeat(qhat(inp["q"].numpy()), 2, axis=2)[:, 0]
    v = inp["v"].numpy()[:, 0]                                  # [B,Hv,D]
    be = inp["beta"].numpy()[:, 0]                              # [B,Hv]
    expect_state = be[:, :, None, None] * v[:, :, :, None] * kh[:, :, None, :]
    expect_o = be[:, :, None] * v * (kh * qh).sum(-1, keepdims=True)
    assert rel_err(st, expect_state) <= 1e-14
    assert rel_err(y[:, 0], expect_o) <= 1e-14


def test_delta_rule_retrieval_beta_one():
    _, inp = small(1, 1, 1, 1, 16, s0_std=0.5, seed=44)
    inp["log_decay"] = torch.zeros_like(inp["log_decay"])
    inp["beta"] = torch.ones_like(inp["beta"])
    inp["q"] = inp["k"].clone()
    y, st = orun(inp, gated=False)
    k = inp["k"].numpy()[0, 0, 0]
    kh = khat(k)
    n = (k * k).sum() / ((k * k).sum() + 1e-6)                # k^ . k^
    s0 = inp["s0"].numpy()[0, 0]
    v = inp["v"].numpy()[0, 0, 0]
    retrieved = st[0, 0] @ kh
    assert rel_err(retrieved, (1 - n) * (s0 @ kh) + n * v) <= 1e-13
    assert rel_err(retrieved, v) <= 1e-6                      # ~v (eps effect only)
    assert rel_err(y[0, 0, 0], retrieved / np.sqrt(16.0)) <= 1e-13


def test_zero_key_gives_pure_decay_step():
    _, inp = small(1, 1, 1, 1, 8, seed=45)
    inp["k"] = torch.zeros_like(inp["k"])
    _, st = orun(inp, gated=False)
    alpha = np.exp(inp["log_decay"].numpy()[0, 0, 0])
    assert np.array_equal(st[0, 0], alpha * inp["s0"].numpy()[0, 0])


def test_state_orientation_row_is_value_index():
    D = 8
    _, inp = small(1, 1, 1, 1, D, seed=46)
    s0 = torch.zeros(1, 1, D, D, dtype=torch.float64)
    s0[0, 0, 5, 2] = 1.0                                       # row 5 (value), column 2 (key)
    inp["s0"] = s0
    inp["log_decay"] = torch.zeros_like(inp["log_decay"])
    inp["beta"] = torch.zeros_like(inp["beta"])
    q = torch.zeros_like(inp["q"])
    q[0, 0, 0, 2] = 1.0
    inp["q"] = q
    y, _ = orun(inp, gated=False)
    expect = np.zeros(D)
    expect[5] = 1.0 / np.sqrt(1.0 + 1e-6) / np.sqrt(D)
    assert rel_err(y[0, 0, 0], expect) <= 1e-15


def test_boundedness_along_a_long_slow_decay_run():
    # ||k^|| <= 1, beta in (0,1), alpha in (0,1]  =>  ||S_new||_2 <= alpha ||S||_2 + beta ||v||
    _, inp = small(1, 40, 1, 2, 16, s0_std=0.02, seed=47, ldr=(-8.0, -3.0))
    S = inp["s0"]
    for t in range(40):
        step = {k: (None if v is None else v) for k, v in inp.items()}
        for name in ("q", "k", "v", "z", "log_decay", "beta"):
            step[name] = inp[name][:, t:t + 1]
        step["s0"] = S
        _, st = orun(step, gated=False)
        for hv in range(2):
            a = np.exp(step["log_decay"].numpy()[0, 0, hv])
            b = step["beta"].numpy()[0, 0, hv]
            lhs = np.linalg.norm(st[0, hv], 2)
            rhs = a * np.linalg.norm(S.numpy()[0, hv], 2) + b * np.linalg.norm(
                step["v"].numpy()[0, 0, hv])
            assert lhs <= rhs * (1 + 1e-12)
        S = torch.from_numpy(st)


# ------------------------------------------------------------------ exact invariances

@pytest.mark.parametrize("mode", ["literal", "fused"])
def test_power_of_two_scaling_is_exact(mode):
    _, inp = small(2, 6, 2, 4, 8, seed=51)
    y, st = orun(inp, gated=False, mode=mode)
    inp2 = dict(inp)
    inp2["v"] = inp["v"] * 4.0
    inp2["s0"] = inp["s0"] * 4.0
    y2, st2 = orun(inp2, gated=False, mode=mode)
    assert np.array_equal(y2, 4.0 * y)
    assert np.array_equal(st2, 4.0 * st)
    # gated output: scaling o by 4 changes only the weight of the norm eps, so y is scaled
    # by one factor per (b, t, hv) row, and that factor is >= 1 (eps matters less).
    yg, _ = orun(inp, gated=True, mode=mode)
    yg2, _ = orun(inp2, gated=True, mode=mode)
    ratio = yg2 / yg
    assert np.max(np.abs(ratio / ratio[..., :1] - 1.0)) <= 1e-12
    assert np.all(ratio[..., 0] >= 1.0)


def test_query_and_key_scale_invariance():
    _, inp = small(1, 6, 1, 2, 16, seed=52)
    y, st = orun(inp, gated=False)
    inp2 = dict(inp)
    inp2["q"] = inp["q"] * 3.0
    inp2["k"] = inp["k"] * 0.5
    y2, st2 = orun(inp2, gated=False)
    assert rel_err(y2, y) <= 1e-5 and rel_err(st2, st) <= 1e-5   # eps only


def test_key_dim_permutation():
    _, inp = small(1, 5, 2, 4, 8, seed=53)
    P = torch.randperm(8, generator=torch.Generator().manual_seed(1))
    y, st = orun(inp, gated=False)
    inp2 = dict(inp)
    inp2["q"] = inp["q"][..., P]
    inp2["k"] = inp["k"][..., P]
    inp2["s0"] = inp["s0"][..., P]
    y2, st2 = orun(inp2, gated=False)
    assert rel_err(y2, y) <= 1e-13
    assert rel_err(st2, st[..., P.numpy()]) <= 1e-13


def test_value_dim_permutation():
    _, inp = small(1, 5, 2, 4, 8, seed=54)
    P = torch.randperm(8, generator=torch.Generator().manual_seed(2))
    y, st = orun(inp, gated=True)
    inp2 = dict(inp)
    inp2["v"] = inp["v"][..., P]
    inp2["z"] = inp["z"][..., P]
    inp2["gn"] = inp["gn"][P]
    inp2["s0"] = inp["s0"][:, :, P, :]
    y2, st2 = orun(inp2, gated=True)
    Pn = P.numpy()
    assert rel_err(y2, y[..., Pn]) <= 1e-13
    assert rel_err(st2, st[:, :, Pn, :]) <= 1e-13


def test_value_heads_within_group_and_key_groups_permutation():
    # Hk=2 key groups of 2 value heads: value head hv uses key head hv // 2.
    _, inp = small(1, 5, 2, 4, 8, seed=55)
    y, st = orun(inp, gated=True)
    for vperm, kperm in (([1, 0, 3, 2], [0, 1]), ([2, 3, 0, 1], [1, 0]),
                         ([3, 2, 0, 1], [1, 0])):
        inp2 = dict(inp)
        vp, kp = torch.tensor(vperm), torch.tensor(kperm)
        for name in ("v", "z"):
            inp2[name] = inp[name][:, :, vp]
        for name in ("log_decay", "beta"):
            inp2[name] = inp[name][:, :, vp]
        inp2["q"] = inp["q"][:, :, kp]
        inp2["k"] = inp["k"][:, :, kp]
        inp2["s0"] = inp["s0"][:, vp]
        y2, st2 = orun(inp2, gated=True)
        assert np.array_equal(y2, y[:, :, vperm]), (vperm, kperm)
        assert np.array_equal(st2, st[:, vperm])


# ------------------------------------------------------------------------ compositions

def test_split_scan_equals_single_scan():
    _, inp = small(2, 9, 2, 4, 8, seed=61)
    y, st = orun(inp)
    first = dict(inp)
    second = dict(inp)
    for name in ("q", "k", "v", "z", "log_decay", "beta"):
        first[name] = inp[name][:, :4]
        second[name] = inp[name][:, 4:]
    y1, st1 = orun(first)
    second["s0"] = torch.from_numpy(st1)
    y2, st2 = orun(second)
    assert np.array_equal(np.concatenate([y1, y2], axis=1), y)
    assert np.array_equal(st2, st)


def _transition_and_offset(inp, lo, hi):
    """M (Dk x Dk, the memory the identity becomes with v = 0) and N (the end memory from
    zeros) of tokens [lo, hi), both from the oracle."""
    seg = {k: (v[:, lo:hi].contiguous() if k in ("q", "k", "v", "z", "log_decay", "beta") else v)
           for k, v in inp.items()}
    B, S, _, Dk = seg["q"].shape
    Hv = seg["v"].shape[2]
    _, N = orun(dict(seg, s0=None), gated=False)
    ident = dict(seg, v=torch.zeros(B, S, Hv, Dk, dtype=torch.float64),
                 s0=torch.eye(Dk, dtype=torch.float64).expand(B, Hv, Dk, Dk).contiguous())
    _, M = orun(ident, gated=False)
    return M, N


def test_segment_end_memory_is_an_affine_map_of_its_start():
    # The update is affine in the memory (codegen_cuda::gdn, "The fusion"), so a segment of
    # tokens maps its start memory S0 to S0 M + N.  This is the identity the sequence-split
    # scan composes; checked on the oracle alone, with Dk != Dv, grouped heads, one segment and
    # a chain of two.
    _, inp = small(2, 7, 2, 4, 6, seed=62, Dk=5, Dv=6)
    _, s_end = orun(inp, gated=False)
    s0 = inp["s0"].numpy()
    M, N = _transition_and_offset(inp, 0, 7)
    assert M.shape == (2, 4, 5, 5) and N.shape == s0.shape
    assert rel_err(s0 @ M + N, s_end) <= 1e-12
    M1, N1 = _transition_and_offset(inp, 0, 3)
    M2, N2 = _transition_and_offset(inp, 3, 7)
    assert rel_err((s0 @ M1 + N1) @ M2 + N2, s_end) <= 1e-12
    # M contracts (each factor alpha (I - beta k^ k^T) has spectral norm <= 1)
    assert np.all(np.linalg.norm(M, ord=2, axis=(-2, -1)) <= 1 + 1e-12)


def test_decode_steps_equal_scan():
    _, inp = small(1, 6, 1, 2, 8, seed=62)
    y, st = orun(inp)
    S = inp["s0"]
    for t in range(6):
        step = dict(inp)
        for name in ("q", "k", "v", "z", "log_decay", "beta"):
            step[name] = inp[name][:, t:t + 1]
        step["s0"] = S
        yt, S = orun(step)
        assert np.array_equal(yt[:, 0], y[:, t])
        S = torch.from_numpy(S)
    assert np.array_equal(S.numpy(), st)


def test_head_major_equals_seq_major():
    _, inp = small(2, 5, 2, 4, 8, seed=63)
    y, st = orun(inp)
    hm = dict(inp)
    for name in ("q", "k", "v", "z"):
        hm[name] = inp[name].transpose(1, 2).contiguous()
    for name in ("log_decay", "beta"):
        hm[name] = inp[name].transpose(1, 2).contiguous()
    y2, st2 = orun(hm, head_major=True)
    assert np.array_equal(y2, y.transpose(0, 2, 1, 3))
    assert np.array_equal(st2, st)


def test_gqa_equals_explicit_repeat():
    _, inp = small(1, 5, 2, 8, 8, seed=64)
    y, st = orun(inp)
    rep = dict(inp)
    rep["q"] = inp["q"].repeat_interleave(4, dim=2)
    rep["k"] = inp["k"].repeat_interleave(4, dim=2)
    y2, st2 = orun(rep)
    assert np.array_equal(y2, y) and np.array_equal(st2, st)


def test_head_subset_matches_full_run():
    _, inp = small(2, 4, 2, 4, 8, seed=65)
    y, st = orun(inp, threads=3)
    y2, st2 = orun(inp, heads=[5, 0, 7], threads=2)
    for head in (0, 5, 7):
        b, hv = divmod(head, 4)
        assert np.array_equal(y2[b, :, hv], y[b, :, hv])
        assert np.array_equal(st2[b, hv], st[b, hv])
    assert np.isnan(y2[0, :, 1]).all()


def test_threads_do_not_change_results():
    _, inp = small(2, 4, 2, 4, 16, seed=66)
    y1, s1 = orun(inp, threads=1)
    y2, s2 = orun(inp, threads=5)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


# ------------------------------------------------------------------------- gated norm

def test_gated_norm_matches_torch_rmsnorm_and_silu():
    _, inp = small(2, 5, 2, 4, 16, seed=71)
    y_raw, _ = orun(inp, gated=False)
    y, _ = orun(inp, gated=True)
    o = torch.from_numpy(y_raw)
    x = o * torch.nn.functional.silu(inp["z"])
    expect = torch.nn.functional.rms_norm(x, (16,), eps=1e-6) * inp["gn"]
    assert rel_err(y, expect.numpy()) <= 1e-13


# ----------------------------------------------------------------------- edge cases

def test_empty_sequence_copies_initial_state():
    _, inp = small(1, 0, 1, 2, 8, seed=72)
    y, st = orun(inp)
    assert y.shape == (1, 0, 2, 8)
    assert np.array_equal(st, inp["s0"].numpy())


def test_empty_batch():
    _, inp = small(0, 3, 1, 2, 8, seed=73)
    y, st = orun(inp)
    assert y.size == 0 and st.size == 0


def test_bad_arguments_rejected():
    _, inp = small(1, 2, 2, 3, 8, seed=74)       # Hv % Hk != 0
    with pytest.raises(ValueError):
        orun(inp)
