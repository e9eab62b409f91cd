"""fp64 CPU oracle of the implicit-integration hot path (test infrastructure).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
use this package.  The CUDA library never imports, links or calls it.
"""
