"""Per-workload results table: merges the bench lines of the five workloads
(``python bench.py --workload NAME``, one JSON file each) with the parity
statistics the GPU parity test records (``NVFP4KV_PARITY_STATS=path``) into
profiles/results.json and profiles/results.md.

    python tests/results_table.py --bench DIR --parity FILE

DIR holds ``<workload>.json`` files (the bench's JSON line).  Floating-point
operations of the prefix-cache extend workload are counted per visible key:
2 (Dk + Dv) per (query row, head, key)."""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W  # noqa: E402


def flops(batch) -> float:
    c = batch.cfg
    total = 0
    for L in batch.kv_lens:
        for i in range(c.qo_len):
            vis = (L - c.qo_len + i + 1) if c.causal else L
            total += vis * c.num_qo_heads * 2 * (c.head_dim_qk + c.head_dim_vo)
    return float(total)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--bench", required=True)
    ap.add_argument("--parity", required=True)
    ap.add_argument("--out", default=os.path.join(ROOT, "profiles", "results"))
    args = ap.parse_args()
    parity = json.load(open(args.parity))
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    rows = []
    for name in W.WORKLOADS:
        f = os.path.join(args.bench, name + ".json")
        if not os.path.exists(f):
            continue
        b = json.loads(open(f).read().strip().splitlines()[-1])
        batch = W.make_batch(W.WORKLOADS[name])
        us = b["config"]["us_per_call"]
        fl = flops(batch)
        row = {
            "workload": name, "kernel": b["config"]["kernel"],
            "us_per_call": us, "us_spread": b["config"].get("us_per_call_spread"),
            "kv_tokens_per_s": b["value"],
            "algorithmic_bytes": b["config"]["algorithmic_bytes_per_call"],
            "hbm_gbs": b["roofline"]["achieved"], "hbm_frac": b["roofline"]["frac"],
            "gflop": fl / 1e9, "tflops": fl / (us * 1e-6) / 1e12,
            "tensor_frac_bf16": fl / (us * 1e-6) / 1e12 / peaks["bf16_tflops"],
            "e2e_ms": b["e2e"]["ms_per_step"], "clocks": b.get("clocks"),
            "parity": parity.get(name),
        }
        rows.append(row)
    json.dump({"peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"]},
               "rows": rows}, open(args.out + ".json", "w"), indent=1)
    lines = ["| workload | kernel | us/call (median) | KV tokens/s | HBM GB/s | HBM frac | "
             "TFLOP/s | bf16 frac | e2e ms | out max-abs beyond bf16 rounding | lse max-abs | "
             "alpha | NaN |", "|" + "---|" * 13]
    for r in rows:
        pa = r["parity"] or {}
        med = (r["us_spread"] or {}).get("median", r["us_per_call"])
        lines.append("| %s | %s | %.1f (%.1f) | %.3g | %.0f | %.3f | %.1f | %.3f | %.4f | %s | %s | %s "
                     "| %s |" % (r["workload"], r["kernel"], r["us_per_call"], med,
                                 r["kv_tokens_per_s"], r["hbm_gbs"], r["hbm_frac"], r["tflops"],
                                 r["tensor_frac_bf16"], r["e2e_ms"],
                                 "%.2e" % pa["max_abs_beyond_bf16_rounding"] if pa else "-",
                                 "%.2e" % pa["lse_max_abs"] if pa else "-",
                                 "%.5f" % pa["alpha"] if pa else "-",
                                 pa.get("nan", "-") if pa else "-"))
    open(args.out + ".md", "w").write("\n".join(lines) + "\n")
    print("\n".join(lines))


if __name__ == "__main__":
    main()
