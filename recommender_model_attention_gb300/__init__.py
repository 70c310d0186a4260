"""GB300-native GDPA (Generalized Dot-Product Attention) for jagged batches.

    O_b = act(alpha * Q_b K_b^T) V_b   for every sample b and head,

with an element-wise activation in place of softmax (GELU-erf, GELU-tanh,
SiLU, the ALU-only 6th-order Taylor GELU) and no row normalisation, over
jagged batches given by offset arrays, forward and backward.  The work runs
in a C-ABI shared library of hand-written sm_103a CUDA kernels
(``include/gdpa.h``); this package is its ctypes binding.
"""

from .gdpa import (  # noqa: F401
    ACT,
    BLOCK_M,
    BLOCK_N,
    GdpaError,
    LIB_PATH,
    MASK,
    MX,
    Plan,
    STATUS,
    allreduce_seed_grad,
    act_eval,
    gdpa_bwd,
    gdpa_bwd_mx,
    gdpa_fwd,
    gdpa_fwd_mx,
    gdpa_fwd_noalloc,
    gdpa_softmax_bwd,
    gdpa_softmax_fwd,
    lib,
    mx_dequantise,
    mx_quantise,
    shard_batch,
    shard_rows,
)


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree for sm_103a; returns its path."""
    from ._build import build as _b
    return _b(force=force)
