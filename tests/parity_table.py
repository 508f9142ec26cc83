"""Turn the margins the full-size parity tests record into a markdown table.

The full-size parity tests append one JSON line per case to the file named by the
``GDN_PARITY_LOG`` environment variable: the workload, the kernel, the output compared (gated y
or raw o), max |gpu - oracle| / (1 + |oracle|) on y and on the final state, and the tolerance.

    GDN_PARITY_LOG=/tmp/margins.jsonl python -m pytest tests -m gpu
    python tests/parity_table.py /tmp/margins.jsonl <output table> "<command>"
"""
from __future__ import annotations

import json
import sys


def table(records: list[dict]) -> str:
    rows = ["| workload | kernel | output | max err y | max err state | tolerance | "
            "worst / tolerance |",
            "|---|---|---|---|---|---|---|"]
    for r in records:
        worst = max(r["err_y"], r["err_state"])
        rows.append(f"| {r['workload']} | {r['kernel']} | {r['output']} | {r['err_y']:.3e} | "
                    f"{r['err_state']:.3e} | {r['tol']:.0e} | {worst / r['tol']:.4f} |")
    return "\n".join(rows)


def main(argv):
    src, out = argv[1], argv[2]
    command = argv[3] if len(argv) > 3 else ""
    records, seen = [], set()
    for line in open(src):
        line = line.strip()
        if not line:
            continue
        r = json.loads(line)
        key = (r["workload"], r["kernel"], r["output"])
        if key in seen:              # a later run of the same case replaces the earlier one
            records = [x for x in records if (x["workload"], x["kernel"], x["output"]) != key]
        seen.add(key)
        records.append(r)
    text = ["# Parity margins of the full-size cases",
            "",
            "Errors are max |gpu - oracle| / (1 + |oracle|) over every element of y and of the "
            "final state, against the fp64 oracle on the same seeded inputs.",
            ""]
    if command:
        text += [f"Command: `{command}`", ""]
    text += [table(records), ""]
    with open(out, "w") as f:
        f.write("\n".join(text))


if __name__ == "__main__":
    main(sys.argv)
