"""Summarise a parity report (the JSON lines the GPU tests append to $FA_PARITY_REPORT) as a
Markdown table: the named workloads' element-by-element comparison with the oracle (literal max
and mean |err|, the rounding floor, rows compared, the readings asserted), then the backward's
gradient errors.

    FA_PARITY_REPORT=parity.jsonl python -m pytest tests -m gpu
    python tests/parity_report.py parity.jsonl > summary.md
"""
import json
import sys
from pathlib import Path

sys.path.insert(0, str(Path(__file__).resolve().parent.parent))
from tiled_online_softmax_gb300 import inputs  # noqa: E402

NAMED = ("single_head", "ragged", "causal_prefill", "rescale_stress", "long_causal", "headline",
         "headline_d64")


def main(path: str) -> None:
    recs = [json.loads(line) for line in open(path) if line.strip()]
    def shape(w):
        return (f"B={w.B} H={w.H} Nq={w.Nq} Nk={w.Nk} D={w.D} {w.dtype}"
                f"{' causal' if w.causal else ''}")

    fwd = {}
    for r in recs:
        # the full-size comparison of each named workload, at its own shape
        if r.get("what") in NAMED and r.get("shape") == shape(inputs.WORKLOADS[r["what"]]):
            fwd[r["what"]] = r
    print("| workload | shape | rows compared | max abs err | mean abs err | rounding floor (max) |"
          " rounding floor (mean) | max reading | mean reading (bound) | oracle on the host |")
    print("|---|---|---|---|---|---|---|---|---|---|")
    for name in NAMED:
        r = fwd.get(name)
        if r is None:
            continue
        host = (f"{r['oracle_seconds']:.2f} s, {r['oracle_threads']} threads"
                if "oracle_seconds" in r else "")
        print(f"| {name} | {r['shape']} | {r['rows']:,} | {r['max_err']:.3e} | {r['mean_err']:.3e} |"
              f" {r['rounding_floor']:.3e} | {r['mean_floor']:.2e} | {r['max_reading']} |"
              f" {r['mean_reading']} ({r['mean_bound']:.2e}) | {host} |")
    for r in recs:
        if str(r.get("what", "")).endswith("fp32 output"):
            print(f"\n{r['what']} ({r['shape']}, every element, O written in fp32 before rounding): "
                  f"max abs err {r['max_err']:.3e}, mean {r['mean_err']:.3e}, against the literal "
                  f"1e-2 and 1e-3.")
    others = [r for r in recs if "rel_norm_err" not in r
              and fwd.get(r.get("what")) is not r and not str(r.get("what", "")).endswith("fp32 output")]
    if others:
        worst = max(others, key=lambda r: r["mean_err"] / r["mean_bound"])
        unshaped = sum(1 for r in others if not r.get("shape"))
        within = all(r["worst_excess"] <= 0 and r["mean_err"] <= r["mean_bound"] for r in others)
        print(f"\nOther comparisons: {len(others)} (edge shapes, negative and zero scale, rising "
              f"maxima, lazy-rescale thresholds, split over keys, rotary inputs, LSE cases, "
              f"streams and graphs; {unshaped} recorded without their shape). Largest mean |err| "
              f"relative to its bound: {worst['what']} ({worst.get('shape') or 'shape not recorded'}), "
              f"mean {worst['mean_err']:.3e} against {worst['mean_bound']:.2e} "
              f"({worst['mean_reading']}); largest max |err| of them: "
              f"{max(r['max_err'] for r in others):.3e}; "
              f"{'every one within its bar' if within else 'NOT all within their bars'}.")
    bwd = [r for r in recs if "rel_norm_err" in r]
    if bwd:
        print("\n| backward gradient | shape | elements | norm error / norm | max error / largest magnitude |")
        print("|---|---|---|---|---|")
        for r in bwd:
            print(f"| {r['what']} | {r['shape']} | {r['elements']:,} | {r['rel_norm_err']:.3e} |"
                  f" {r['rel_max_err']:.3e} |")


if __name__ == "__main__":
    main(sys.argv[1])
