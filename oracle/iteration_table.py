"""Record how many PCG iterations the fp64 oracle needs on the first step of
each named configuration (test infrastructure).

The benchmark's CPU baseline times the oracle on a bounded sample (one
assembly plus a few PCG iterations) and extrapolates to a whole step with the
counts stored here.  Only the oracle and the seeded input generators run.

    python -m oracle.iteration_table C1 C2 C3 C4 C5
"""
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

from oracle import oracle  # noqa: E402
from sparse_linear_solve_gb300 import workloads as W  # noqa: E402

TABLE = os.path.join(HERE, "iteration_table.json")


def main(names):
    table = {}
    if os.path.exists(TABLE):
        with open(TABLE) as f:
            table = json.load(f)
    for name in names:
        w = W.make(name)
        c = w.contacts(0)
        t0 = time.perf_counter()
        s = oracle.assemble_workload(w, w.x0, w.v0, c if c.n else None)
        dv, it, rr, st = s.pcg(w.tol, w.maxit)
        table[name] = dict(iterations=[it], relres=[rr], status=[st], steps=[0],
                           tol=w.tol, seconds=time.perf_counter() - t0)
        print(name, table[name], flush=True)
        with open(TABLE, "w") as f:
            json.dump(table, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or ["C1", "C2", "C3", "C4", "C5"])
