"""The five scan workloads, by name, with their sizes.

Each entry gives the problem as the library's ``ssd_problem`` describes it:
variant ('mamba2' | 'mamba1' | 'mimo'), io dtype ('f32' | 'bf16'), batch,
seqlen T, nheads H (channels D for Mamba-1), headdim P (1 for Mamba-1),
dstate N, ngroups G, chunk length L and mimo_rank R.
"""
from __future__ import annotations

CONFIGS = {
    # tiny Mamba-2 scan in fp32; the oracle finishes it in milliseconds
    "mamba2_tiny_fp32": dict(variant="mamba2", dtype="f32", batch=1, seqlen=64, nheads=2, headdim=8,
                             dstate=4, ngroups=1, chunk=16, mimo_rank=1),
    # Mamba-2 130M layer shape
    "mamba2_130m_bf16": dict(variant="mamba2", dtype="bf16", batch=8, seqlen=2048, nheads=24, headdim=64,
                             dstate=128, ngroups=1, chunk=64, mimo_rank=1),
    # Mamba-2 2.7B layer shape (the headline throughput workload)
    "mamba2_2p7b_bf16": dict(variant="mamba2", dtype="bf16", batch=4, seqlen=4096, nheads=80, headdim=64,
                             dstate=128, ngroups=1, chunk=64, mimo_rank=1),
    # Mamba-1 branch: one decay per state, D channels of width 1
    "mamba1_fp32": dict(variant="mamba1", dtype="f32", batch=8, seqlen=2048, nheads=1536, headdim=1,
                        dstate=16, ngroups=1, chunk=64, mimo_rank=1),
    # Mamba-3 MIMO pass, rank 4 (fused chunk length L*R = 256)
    "mimo_r4_bf16": dict(variant="mimo", dtype="bf16", batch=4, seqlen=4096, nheads=32, headdim=64,
                         dstate=128, ngroups=32, chunk=64, mimo_rank=4),
}

HEADLINE = "mamba2_2p7b_bf16"

# The KDA delta-rule recurrence (a second workload with its own entry points): batch, seqlen T, nheads H (query
# and key heads), value_heads HV (a multiple of H: each query / key head serves HV / H value heads), key_dim K,
# value_dim V, fp32 io.  The pages give no sizes for it; these are a head dimension of 128 and a short context.
KDA_CONFIGS = {
    # tiny; the float64 oracle's finite differences cover every element of it
    "kda_tiny_fp32": dict(variant="kda", dtype="f32", batch=1, seqlen=16, nheads=2, value_heads=4, key_dim=8,
                          value_dim=8),
    # head dimension 128, 16 value heads over 8 query / key heads, T = 1024
    "kda_fp32": dict(variant="kda", dtype="f32", batch=2, seqlen=1024, nheads=8, value_heads=16, key_dim=128,
                     value_dim=128),
}


def tokens(cfg: dict) -> int:
    """Tokens per forward+backward pair: batch x seqlen."""
    return cfg["batch"] * cfg["seqlen"]


def scaled(cfg: dict, **over) -> dict:
    """A copy of ``cfg`` with some sizes replaced (for small parity cases)."""
    out = dict(cfg)
    out.update(over)
    return out
