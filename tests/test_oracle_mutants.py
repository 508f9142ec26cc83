"""Planted mistakes in the oracle must fail its pins (CPU only).

Each case copies ``oracle/gdn_oracle.c`` to a temporary folder, plants one plausible
mistake by a textual edit (a dropped term, a wrong sign, a transposed or wrong index, a
misplaced eps, a missing scale, ...), compiles the copy with the oracle's own flags and runs
a compact battery of pins against it: the 50-digit decimal brute force on small cases in
both layouts, gated and raw, with grouped heads.  The battery must report a failure for
every mutant and none for the unmodified source.
"""
from __future__ import annotations

import os
import shutil

import numpy as np
import pytest
import torch

import oracle
from oracle import closed_form_decimal
from linear_attention_recurrence_gdn_gb300.workloads import TINY, make_inputs

MUTANTS = {
    "drop_alpha_in_prediction": ("beta * (vi - alpha * wk->u[i])", "beta * (vi - wk->u[i])"),
    "wrong_sign_of_correction": ("beta * (vi - alpha * wk->u[i])",
                                 "beta * (vi + alpha * wk->u[i])"),
    "read_transposed_state": ("acc += S[i * Dk + j] * wk->qh[j];",
                              "acc += S[j * Dk + i] * wk->qh[j];"),
    "missing_query_scale": ("/ sqrt(ssq + a->qk_eps) / sqrt((double)Dk)",
                            "/ sqrt(ssq + a->qk_eps)"),
    "gqa_modulo_mapping": ("hk = hv / (a->Hv / a->Hk)", "hk = hv % a->Hk"),
    "eps_outside_sqrt": ("1.0 / sqrt(ssk + a->qk_eps)", "1.0 / (sqrt(ssk) + a->qk_eps)"),
    "sigmoid_sign": ("zi / (1.0 + exp(-zi))", "zi / (1.0 + exp(zi))"),
    "sum_instead_of_mean": ("ss / (double)Dv + a->norm_eps", "ss + a->norm_eps"),
    "norm_weight_index": ("* r * a->gn[i]", "* r * a->gn[0]"),
    "decay_not_exponentiated": ("exp(a->g[idx_gate(a, b, t, hv)])", "(a->g[idx_gate(a, b, t, hv)])"),
    "fused_output_missing_alpha": ("wk->o[i] = alpha * ww + coef * kq;",
                                   "wk->o[i] = ww + coef * kq;"),
    "head_major_query_index": ("return ((b * a->Hk + h) * a->S + t) * a->Dk + j;",
                               "return ((b * a->S + t) * a->Hk + h) * a->Dk + j;"),
    "beta_dropped_from_update": ("S[i * Dk + j] = alpha * S[i * Dk + j] + coef * wk->kh[j];",
                                 "S[i * Dk + j] = alpha * S[i * Dk + j] + (coef / beta) * wk->kh[j];"),
    "initial_state_ignored": ("S[i] = a->s0 ? a->s0[head * Dv * Dk + i] : 0.0;", "S[i] = 0.0;"),
}
# Literal mode reading the OLD memory for o: evaluate o before the update pass and skip the
# update (the page is explicit that o reads the UPDATED memory).
MUTANTS["literal_reads_old_memory"] = (
    "            /* pass 2: S = alpha S + beta (v - alpha u) k^T */",
    "            for (int64_t i = 0; i < Dv; i++) {\n"
    "                double acc = 0.0;\n"
    "                for (int64_t j = 0; j < Dk; j++)\n"
    "                    acc += S[i * Dk + j] * wk->qh[j];\n"
    "                wk->o[i] = acc;\n"
    "            }\n"
    "            if (0)\n"
    "            /* pass 2: S = alpha S + beta (v - alpha u) k^T */")

CASES = [
    # B, S, Hk, Hv, D, head_major, gated, seed
    (1, 3, 2, 4, 4, False, True, 81),
    (1, 3, 2, 4, 4, True, False, 82),
    (2, 2, 1, 2, 4, False, False, 83),
]


def _inputs(case):
    B, S, Hk, Hv, D, hm, gated, seed = case
    w = TINY.replace(name="m", B=B, S=S, Hk=Hk, Hv=Hv, Dk=D, Dv=D, head_major=hm, seed=seed)
    inp = {k: (None if v is None else v.double().numpy()) for k, v in make_inputs(w).items()}
    if not gated:
        inp["z"] = inp["gn"] = None
    return inp


@pytest.fixture(scope="module")
def references():
    refs = []
    for case in CASES:
        inp = _inputs(case)
        refs.append(closed_form_decimal.run(inp["q"], inp["k"], inp["v"], inp["log_decay"],
                                            inp["beta"], z=inp["z"], gn=inp["gn"],
                                            s0=inp["s0"], head_major=case[5]))
    return refs


def battery(library, references) -> list[str]:
    """Return the names of the pins the oracle in ``library`` fails."""
    failures = []
    for case, (yd, sd) in zip(CASES, references):
        inp = _inputs(case)
        for mode in ("literal", "fused"):
            try:
                y, st = oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                                   z=inp["z"], gn=inp["gn"], s0=inp["s0"], head_major=case[5],
                                   mode=mode, library=library)
            except ValueError:
                failures.append(f"{case}:{mode}:rejected")
                continue
            err = max(np.max(np.abs(y - yd) / (1 + np.abs(yd))),
                      np.max(np.abs(st - sd) / (1 + np.abs(sd))))
            if not err <= 1e-12:
                failures.append(f"{case}:{mode}:err={err:.3g}")
    return failures


def _build_variant(tmp_path, name, edit):
    src = open(oracle.SOURCE).read()
    if edit is not None:
        old, new = edit
        assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new, 1)
    d = tmp_path / name
    d.mkdir()
    shutil.copy(os.path.join(os.path.dirname(oracle.SOURCE), "gdn_oracle.h"), d)
    path = d / "gdn_oracle.c"
    path.write_text(src)
    return oracle.compile_oracle(str(path), str(d / "lib.so"))


def test_unmodified_oracle_passes_battery(tmp_path, references):
    lib = _build_variant(tmp_path, "clean", None)
    assert battery(lib, references) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, references, name):
    lib = _build_variant(tmp_path, name, MUTANTS[name])
    assert battery(lib, references), f"mutant {name} passed every pin"
