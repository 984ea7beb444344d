"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This package holds input generation only — random numbers, dtype rounding and
the shapes of the workloads — and none of the attention arithmetic.  Both the
CUDA path's tests/bench and the CPU oracle consume what it returns; it imports
neither of them.
"""

from .gen import (  # noqa: F401
    SEED_BASE,
    TID,
    bf16_bits,
    bf16_bits_to_f64,
    bf16_round,
    normal,
    normal_at,
    normal_device,
    row_softmax_mixing,
    uniform,
    uniform_at,
    uniform_row_normalised_mixing,
)
from .configs import (  # noqa: F401
    WORKLOADS,
    Workload,
    decode_device,
    decode_host,
    make_mixing,
    mhla_device,
    mhla_host,
    rala_device,
    rala_host,
)
