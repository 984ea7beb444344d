"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This package holds input generation only — random numbers, dtype rounding and
the shapes of the workloads — and none of the attention arithmetic.  Both the
CUDA path's tests/bench and the CPU oracle consume what it returns; it imports
neither of them.
"""

from .gen import (  # noqa: F401
    SEED_BASE,
    TID,
    normal,
    uniform,
    bf16_bits,
    bf16_round,
    bf16_bits_to_f64,
    row_softmax_mixing,
    uniform_row_normalised_mixing,
)
from .configs import WORKLOADS, Workload, make_mhla_inputs, make_rala_inputs, make_decode_inputs  # noqa: F401
