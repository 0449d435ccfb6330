"""MiniMax-H3 BF16 pre-attention stage for GB300 (sm_103a).

The stage (input RMSNorm, indexed AdaLN, fused QKV projection, per-head Q/K
RMSNorm, partial split-half RoPE, destination-major pack) runs in two CUDA
kernels behind the C ABI declared in include/mh3_preattn.h.  ``binding``
marshals torch tensors into that ABI; ``inputs`` draws seeded synthetic
workloads; ``build`` compiles the library in-tree.

Importing this package loads nothing; the library is loaded on first use.
"""


def minimax_h3_bf16_pre_attention(*args, **kwargs):
    from .binding import minimax_h3_bf16_pre_attention as _f
    return _f(*args, **kwargs)
