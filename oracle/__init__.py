"""CPU oracle of the MiniMax-H3 BF16 pre-attention stage.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
CPU-baseline / reference arm may import this package.  The product path (the
CUDA library and its Python binding) never imports, calls or links it, and
the oracle shares no code with the CUDA path.

Plain, slow, shape-generic PyTorch CPU code: FP32 elementwise steps with the
BF16 rounding points the pages name, and float64 reductions rounded once to
FP32 (the ideal FP32 accumulator; the pages fix FP32 accumulation but no
summation order).

Pins: every function is pinned by tests that do not re-type its formula
(closed forms, library routines for special cases, exact integer arithmetic,
invariants).  No function here is "parity unpinned".
"""
from .preattn import (  # noqa: F401
    input_rmsnorm,
    indexed_adaln,
    qkv_projection,
    head_rmsnorm,
    rope_cache_rows,
    rope_split_half,
    ulysses_pack,
    ulysses_unpack_rows,
    pre_attention_tokens,
    pre_attention,
    PreAttnTokens,
)
from . import out_proj  # noqa: F401  (attention output projection + gated residual)
from . import mlp  # noqa: F401  (MLP block)
from . import e4m3  # noqa: F401  (e4m3 output mode)
from . import nvfp4  # noqa: F401  (NVFP4 pre-attention)
