"""Writes expected_tokens_per_step.json: E[emitted tokens per verify step] when
each draft is right independently with probability alpha and acceptance stops
at the first wrong draft. Draft j is accepted with probability alpha^j, and the
step always adds the target's own token, so E = sum_{j=0..k} alpha^j =
(1 - alpha^(k+1)) / (1 - alpha). The (alpha, k) pairs are the acceptance
settings of the benchmark workloads."""
import json
import os
from fractions import Fraction

PAIRS = [(0.0, 3), (0.5, 3), (0.8, 3), (0.7, 4), (0.6, 4), (0.5, 4), (0.8, 4)]


def main():
    rows = []
    for a, k in PAIRS:
        fa = Fraction(str(a))
        e = sum(fa ** j for j in range(k + 1))
        rows.append({"alpha": a, "k": k, "expected": float(e)})
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "expected_tokens_per_step.json")
    with open(path, "w") as f:
        json.dump({"rule": "sum_{j=0..k} alpha^j", "rows": rows}, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
