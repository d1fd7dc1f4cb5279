"""CPU oracle of the quantized MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Imported only by the tests, the smoke check and the benchmark's CPU-baseline leg; the
CUDA library never reaches it. ``moe`` is the float64 numpy oracle; ``brute`` is a
pure-Python brute force that pins it on tiny problems.
"""
from . import moe, brute  # noqa: F401
