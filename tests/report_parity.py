"""Writes the parity error table from the statistics the GPU parity tests record.

Run the GPU tests with VP_PARITY_REPORT=<file.json> (tests/conftest.py writes the
statistics there at the end of the session), then

    python -m tests.report_parity <file.json> tests/parity_errors.md

For every bf16 gradient check: elements compared, how many differ from the
oracle's rounded fp64 gradient by more than one bf16 ulp, the worst error in
ulps and the worst error as a fraction of the check's tolerance; for the fused
linear gradients also the worst excess over one ulp relative to the
root-sum-square of the dot product's terms; and the error of the forward's
centred mean c against the oracle's.
"""
import json
import math
import sys


def _family(name: str) -> str:
    if name.endswith(" c"):
        return "forward centred mean c"
    if " dW" in name or "dhidden" in name:
        if "beta=" in name or "JSD" in name:
            return "fused linear JSD"
        if "entropy" in name:
            return "fused linear entropy"
        if "shard" in name:
            return "fused linear, sharded"
        if any(s in name for s in ("Da=", "dir=", "close models", "wide spread")):
            return "fused linear KL"
        return "fused linear logp"
    if name.split()[-1] in ("dA", "dB"):
        return "generalized JSD"
    if name.endswith(" dx") and "K=" in name or name.startswith("full topk"):
        return "top-k"
    if name.startswith("sharded"):
        return "logits, sharded"
    return "logprobs / entropy / KL"


def table(stats: dict) -> str:
    grad = {k: v for k, v in stats.items() if "beyond_1ulp" in v}
    cvals = {k: v for k, v in stats.items() if k.endswith(" c")}
    lines = ["# Parity errors of the GPU tests against the fp64 oracle", "",
             "Written by `tests/report_parity.py` from the statistics the GPU parity tests record "
             "(`VP_PARITY_REPORT`). ulp = one bf16 ulp of the oracle's rounded fp64 gradient; tol = the "
             "check's tolerance (tests/parity.py).", ""]
    fams = {}
    for k, v in grad.items():
        fams.setdefault(_family(k), []).append((k, v))
    lines += ["## Summary by family", "",
              "| family | checks | elements | beyond 1 ulp | share | worst err / tol | κ needed (κ) |",
              "|---|---:|---:|---:|---:|---:|---:|"]
    for fam in sorted(fams):
        rows = fams[fam]
        n = sum(v["n"] for _, v in rows)
        b = sum(v["beyond_1ulp"] for _, v in rows)
        w = max(v.get("worst_over_tol", 0.0) for _, v in rows)
        kn = [v["kappa_needed"] for _, v in rows if "kappa_needed" in v]
        kk = {v["kappa"] for _, v in rows if "kappa" in v}
        ks = f"{max(kn):.2f} ({'/'.join(f'{x:g}' for x in sorted(kk))})" if kn else ""
        lines.append(f"| {fam} | {len(rows)} | {n} | {b} | {b / n if n else 0:.2e} | {w:.3f} | {ks} |")
    lines += ["", "κ needed: the smallest conditioning factor κ in the tolerance term κ·2⁻²⁴·M (tests/parity.py) with "
              "which every element of the family's checks would still pass, every other term of the tolerance "
              "(one ulp, the oracle's rounding, the GEMM's root-sum-square and flush terms) kept; κ: the factor "
              "the checks use."]
    lines += ["", "## Every gradient check", "",
              "| check | elements | beyond 1 ulp | worst err (ulp) | worst err / tol | κ needed | GEMM: worst excess / RSS |",
              "|---|---:|---:|---:|---:|---:|---:|"]
    for k in sorted(grad):
        v = grad[k]
        r = v.get("worst_beyond_ulp_over_rss")
        rs = "" if r is None else ("0" if r <= 0 else f"2^{math.log2(r):.1f}")
        kn = f"{v['kappa_needed']:.2f}" if "kappa_needed" in v else ""
        lines.append(f"| {k} | {v['n']} | {v['beyond_1ulp']} | {v['worst_err_over_ulp']:.3g} | "
                     f"{v.get('worst_over_tol', 0.0):.3f} | {kn} | {rs} |")
    if cvals:
        lines += ["", "## Forward centred mean c of the saved records", "",
                  "| check | rows | max abs error | max rel error |", "|---|---:|---:|---:|"]
        for k in sorted(cvals):
            v = cvals[k]
            lines.append(f"| {k} | {v['n']} | {v['max_abs_err']:.3e} | {v['max_rel_err']:.3e} |")
    return "\n".join(lines) + "\n"


def main(argv):
    if len(argv) != 3:
        print(__doc__)
        return 2
    with open(argv[1]) as f:
        stats = json.load(f)
    with open(argv[2], "w") as f:
        f.write(table(stats))
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
