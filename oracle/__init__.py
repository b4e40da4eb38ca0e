"""fp64 CPU oracle of the routed MoE / LatentMoE layer.

Test infrastructure only: imported by the tests, by the package entry's smoke check and
by the benchmark's CPU-baseline leg, never by the CUDA path.
"""
from . import moe_oracle  # noqa: F401
