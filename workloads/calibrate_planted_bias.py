"""Calibrate beta of the long-context decode workload (b=8, 32768 compressed positions).

One percent of each sequence's index-key rows get `beta * u` added (u: the sequence's
weights-combined index query, unit RMS).  beta is chosen by bisection so that, over the
batch, the median oracle score of the planted rows sits 3 standard deviations (of the
other rows' scores) above the other rows' median.  Only the oracle computes scores here;
the result is written to planted_bias.json beside this file.

    python -m workloads.calibrate_planted_bias
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import workloads  # noqa: E402


def excess_sigma(beta: float) -> float:
    shp = workloads.config(4)
    data = workloads.make(shp, beta=beta)
    score = oracle.index_score(data["iq"], data["ik"], data["w"], shp.index_scale, data["start_pos"], shp.n_cols,
                               shp.ratio)
    zs = []
    for bi in range(shp.b):
        row = score[bi, 0]
        planted = data["planted_rows"][bi]
        mask = np.zeros(row.size, bool)
        mask[planted] = True
        rest = row[~mask]
        zs.append((np.median(row[mask]) - np.median(rest)) / rest.std())
    return float(np.median(zs))


def main():
    lo, hi = 0.0, 4.0
    while excess_sigma(hi) < 3.0:
        hi *= 2
    for _ in range(18):
        mid = 0.5 * (lo + hi)
        if excess_sigma(mid) < 3.0:
            lo = mid
        else:
            hi = mid
    beta = 0.5 * (lo + hi)
    z = excess_sigma(beta)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "planted_bias.json")
    with open(path, "w") as f:
        json.dump({"beta": round(beta, 6), "median_excess_sigma": round(z, 4),
                   "how": "bisection on oracle index scores of the long-context decode workload"}, f, indent=1)
        f.write("\n")
    print(beta, z)


if __name__ == "__main__":
    main()
