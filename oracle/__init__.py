"""CPU oracle for the token-level multi-head linear attention (MHLA) forward path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library and its Python binding) never
imports, calls or links anything here, and this package imports nothing from
the product path; the two share no code.  Inputs come from the caller as plain
arrays (the seeded generators in ``workloads`` produce them).

Everything is computed in float64 from the (already dtype-rounded) inputs,
with numpy ``einsum``/``matmul``/``exp``/``linalg`` as the only library
primitives.  Every function cites the passage of the source pages it follows:

* "MHLA: Restoring Expressivity of Linear Attention via Token-Level
  Multi-Head" (paper notes; cited as *MHLA paper* with its section numbers),
* "Linear Attention（线性注意力）笔记" (cited as *Linear Attention notes*),
* "4. Attention" (tutorial; cited as *Attention tutorial*),
* "Breaking the Low-Rank Dilemma of Linear Attention" (CVPR 2025 paper
  notes; cited as *RALA notes*).

Pin status (what fixes each function independently of itself) is listed in
``PIN_STATUS``; the pins live in ``tests/test_oracle_pins.py``.  No function
here is "parity unpinned".
"""

from .mhla_oracle import (  # noqa: F401
    PIN_STATUS,
    phi,
    block_of,
    mhla_block_form,
    mhla_token_expansion,
    mhla_attention_matrix,
    global_linear_attention,
    causal_recurrent,
    causal_chunked,
    causal_bruteforce,
    causal_mhla_chunked,
    causal_mhla_bruteforce,
    decode_steps,
    decayed_causal_bruteforce,
    phi_relu,
    phi_exp,
    FEATURE_MAPS,
    mhla_block_form_feature,
    mhla_token_expansion_feature,
    causal_variant_recurrent,
    causal_variant_bruteforce,
    mhla_block_form_unnormalized,
    grid_block_ids,
    mhla_block_form_ids,
    mhla_token_expansion_ids,
    locality_mixing_init,
    causal_mhla_stream,
    rala_forward,
    rala_bruteforce,
    numerical_rank,
    phi_grad,
    mhla_block_form_backward,
)
