"""CPU oracle for speculative verify / accept / rollback on GatedDeltaNet layers, and for the
hybrid's attention layers in the verify step (KV append + causal attention, KV truncation).

Test infrastructure only: tests, the smoke check and the bench's CPU-baseline leg use it; the
library never does. See oracle.c for what each function computes and which page it follows.
"""
from .oracle import (  # noqa: F401
    OracleDims,
    verify,
    rollback,
    argmax,
    accept_greedy,
    accept_sample,
    accept_tree,
    exp2_spec,
    scale_c,
    weights,
    philox4x32_10,
    draw,
    accept_stats,
    adaptive_enabled,
    AttnDims,
    attn_verify,
    attn_truncate,
    set_threads,
)
