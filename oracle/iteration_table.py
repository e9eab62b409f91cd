"""Record how many PCG iterations the fp64 oracle needs per step of each named
configuration along its own trajectory (test infrastructure).

Step t starts from the oracle's state after step t-1 (x and v updated with
the oracle's own dv) with that step's contact list, as the benchmark's steps
do on the GPU.  The benchmark's reference arm times the oracle on a bounded
sample (one assembly plus a few PCG iterations) and scales it to each step
with the counts stored here.  Only the oracle and the seeded input
generators run.

    python -m oracle.iteration_table [--steps S] C1 C2 C3 C4 C5
"""
import argparse
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

from oracle import oracle  # noqa: E402
from sparse_linear_solve_gb300 import workloads as W  # noqa: E402

TABLE = os.path.join(HERE, "iteration_table.json")


def main(names, steps):
    table = {}
    if os.path.exists(TABLE):
        with open(TABLE) as f:
            table = json.load(f)
    for name in names:
        w = W.make(name)
        x, v = w.x0, w.v0
        its, rrs, sts, secs = [], [], [], []
        for t in range(steps):
            c = w.contacts(t)
            t0 = time.perf_counter()
            res = oracle.step(w, x, v, c if c.n else None)
            secs.append(time.perf_counter() - t0)
            its.append(int(res["iterations"]))
            rrs.append(float(res["relres"]))
            sts.append(int(res["status"]))
            x, v = res["x"].astype(np.float32), res["v"].astype(np.float32)
            table[name] = dict(iterations=its, relres=rrs, status=sts, steps=list(range(len(its))),
                               tol=w.tol, seconds=secs)
            print(name, t, its[-1], "%.1f s" % secs[-1], flush=True)
            with open(TABLE, "w") as f:
                json.dump(table, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--steps", type=int, default=1)
    ap.add_argument("names", nargs="*", default=["C1", "C2", "C3", "C4", "C5"])
    a = ap.parse_args()
    main(a.names, a.steps)
