"""fp64 CPU oracle for the Gated Subspace Inference (GSI) linear map.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (the CUDA library in ``gated_rank_subspace_gsi_gb300`` and its binding)
never imports, links or calls it, and shares no code with it.

Citations "[GSI ...]" refer to the page "Technical summary: Gated Subspace
Inference for transformer acceleration".  The arithmetic lives in
``gsi_oracle.c`` (plain fp64 loops in the page's order); ``oracle.py`` only
marshals numpy arrays into it.

Every function is pinned by ``tests/test_oracle_pins.py`` to facts that the
page and the mathematics fix (hand-derived closed forms, exact rational
brute force, library special cases, Theorem 4), and
``tests/test_oracle_mutants.py`` checks that those pins catch planted
mistakes.  No function is left unpinned.
"""
from .oracle import (  # noqa: F401
    LIB_PATH,
    SRC_PATH,
    OracleLib,
    bf16_decode,
    bf16_encode,
    build,
    default,
    forward,
    forward_bf16,
    num_threads,
    precompute_M,
    precompute_M_bf16,
    spectral_norm,
)
