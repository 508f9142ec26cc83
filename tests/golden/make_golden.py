"""Write the golden fixtures of this folder.  Calls only ``oracle/`` (its decimal brute force).

The pages print no worked example for the recurrence, so the fixtures are tiny cases whose
expected values come from the 50-digit closed-form brute force in
``oracle/closed_form_decimal.py`` (logicaffeine ``codegen_cuda::gdn``, module description:
u = S k, S = alpha S + beta (v - alpha u) k^T, o = S q, o = rmsnorm(o * silu(z)) GN).
Inputs are drawn by the seeded generator and stored in the file as exact hex floats, so the
fixture does not depend on any random-number library.

Run from the repository root:  python tests/golden/make_golden.py
"""
from __future__ import annotations

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from linear_attention_recurrence_gdn_gb300.workloads import TINY, make_inputs  # noqa: E402
from oracle import closed_form_decimal  # noqa: E402

CITATION = ("logicaffeine_compile::codegen_cuda::gdn, module description (the per-token "
            "recurrence and the gated norm); torch_to_nnef.op.gated_delta, "
            "emit_native_gdn_recurrent (operand layouts and head_major) and "
            "native_gdn_reject_reason (q/k l2-norm, 1/sqrt(head_dim) scale)")

CASES = [
    # name, B, S, Hk, Hv, D, head_major, gated, with_s0, seed
    ("seq_major_gated_s0_b1_s3_h1_d4", 1, 3, 1, 1, 4, False, True, True, 11),
    ("head_major_raw_gqa2_b1_s4_hk1_hv2_d4", 1, 4, 1, 2, 4, True, False, False, 12),
    ("seq_major_gated_gqa2_b2_s2_hk2_hv4_d8", 2, 2, 2, 4, 8, False, True, True, 13),
]


def _pack(a) -> dict:
    a = np.asarray(a, dtype=np.float64)
    return {"shape": list(a.shape), "hex": [float(x).hex() for x in a.reshape(-1)]}


def make_case(name, B, S, Hk, Hv, D, head_major, gated, with_s0, seed):
    w = TINY.replace(name=name, B=B, S=S, Hk=Hk, Hv=Hv, Dk=D, Dv=D, head_major=head_major,
                     s0_std=0.1 if with_s0 else None, seed=seed)
    inp = make_inputs(w)
    f64 = {kk: (None if vv is None else vv.double().numpy()) for kk, vv in inp.items()}
    z = f64["z"] if gated else None
    gn = f64["gn"] if gated else None
    y, state = closed_form_decimal.run(f64["q"], f64["k"], f64["v"], f64["log_decay"],
                                       f64["beta"], z=z, gn=gn, s0=f64["s0"],
                                       head_major=head_major, qk_eps=1e-6, norm_eps=1e-6)
    inputs = {"q": f64["q"], "k": f64["k"], "v": f64["v"], "log_decay": f64["log_decay"],
              "beta": f64["beta"]}
    if gated:
        inputs["z"] = z
        inputs["gn"] = gn
    if with_s0:
        inputs["s0"] = f64["s0"]
    return {
        "name": name,
        "citation": CITATION,
        "generated_by": "tests/golden/make_golden.py via oracle/closed_form_decimal.py "
                        "(50 significant digits, rounded to double)",
        "shape": {"B": B, "S": S, "Hk": Hk, "Hv": Hv, "Dk": D, "Dv": D},
        "head_major": head_major,
        "qk_eps": 1e-6,
        "norm_eps": 1e-6,
        "inputs": {kk: _pack(vv) for kk, vv in inputs.items()},
        "expected": {"y": _pack(y), "state": _pack(state)},
    }


def main():
    for case in CASES:
        data = make_case(*case)
        path = os.path.join(HERE, f"gdn_{case[0]}.json")
        with open(path, "w") as f:
            json.dump(data, f, separators=(",", ":"))
            f.write("\n")
        print("wrote", path)


if __name__ == "__main__":
    main()
