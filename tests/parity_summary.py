"""Turn the parity records of a GPU test run into the markdown table kept in
profiles/.

    GNA_PARITY_RECORD=parity.jsonl python -m pytest tests -m gpu
    python tests/parity_summary.py parity.jsonl > profiles/parity_all_configs.md

Each record is one comparison of the CUDA path with the oracle (written by
``tests.gpu_helpers.record_parity``): the forward's max |dout|, max |dlse| and
relative RMS of out, or one gradient's max |error|, its largest reference value
and relative RMS.
"""
from __future__ import annotations

import json
import sys


def _geom(r) -> str:
    if "dims" not in r:
        return ""
    x = lambda v: "x".join(map(str, v))  # noqa: E731
    d = f", d={r['head_dim']}" if "head_dim" in r else ""
    return f"{x(r['dims'])} w {x(r['window'])} s {x(r['stride'])}, {r.get('heads', '?')} heads, B={r.get('B', '?')}{d}"


def main(path: str) -> None:
    recs = [json.loads(line) for line in open(path) if line.strip()]
    fwd = [r for r in recs if r["kind"] == "forward"]
    bwd = [r for r in recs if r["kind"] == "backward"]
    print("| test | geometry | dtype | seed | queries | max abs dout | max abs dlse | rel RMS out |")
    print("|---|---|---|---|---|---|---|---|")
    for r in fwd:
        name = r["test"].split("::")[-1]
        print(f"| `{name}` | {_geom(r)}{' (sampled)' if r.get('sampled') else ''} | {r.get('dtype', '')} | "
              f"{r.get('seed', '')} | {r['n_queries']} | {r['max_abs_out']:.2e} | {r['max_abs_lse']:.2e} | "
              f"{r['rel_rms_out']:.2e} |")
    print()
    print("| test | geometry | seed | gradient | max abs error | max abs gradient | rel RMS |")
    print("|---|---|---|---|---|---|---|")
    for r in bwd:
        name = r["test"].split("::")[-1]
        print(f"| `{name}` | {_geom(r)}{' (sampled)' if r.get('sampled') else ''} | {r.get('seed', '')} | "
              f"{r['grad']} | {r['max_abs_err']:.2e} | {r['max_abs_ref']:.2e} | {r['rel_rms']:.2e} |")
    if fwd:
        bf = [r["rel_rms_out"] for r in fwd if r.get("dtype") == "bf16"]
        f8 = [r["rel_rms_out"] for r in fwd if r.get("dtype") == "fp8"]
        print()
        print(f"Largest relative RMS of out: bf16 {max(bf):.2e} over {len(bf)} configurations"
              + (f", e4m3 {max(f8):.2e} over {len(f8)}" if f8 else "") + ".")
    if bwd:
        print(f"Largest relative RMS of a gradient: {max(r['rel_rms'] for r in bwd):.2e}; largest error "
              f"{100 * max(r['max_abs_err'] / r['max_abs_ref'] for r in bwd):.2f} % of the largest gradient.")


if __name__ == "__main__":
    main(sys.argv[1])
