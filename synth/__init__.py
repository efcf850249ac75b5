"""Seeded synthetic inputs for tree verification (shared by the oracle tests,
the GPU parity tests and the benchmark).

This package only *creates* inputs: tree shapes, tokens, bf16 query/key/value
values, a shuffled paged KV pool with its block table, partial-KV page lists
and logits with a planted accepted path.  It holds none of the verification
arithmetic (no attention, no argmax, no acceptance walk, no commit); the
draft distributions it makes for stochastic acceptance are inputs, built its
own way.
"""

from .workloads import (  # noqa: F401
    CONFIGS,
    VerifyCase,
    bf16_bits_from_f32,
    make_case,
    make_sampling_inputs,
    tree_chain,
    tree_eagle_static,
    tree_random_depth,
    tree_specblock,
    node_depths,
)
