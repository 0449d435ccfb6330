"""CPU oracle of the MiniMax-H3 BF16 pre-attention stage.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
CPU-baseline / reference arm may import this package.  The product path (the
CUDA library and its Python binding) never imports, calls or links it, and
the oracle shares no code with the CUDA path.

The stage's oracle is plain C++ (``cpp/mh3_oracle.cpp``, compiled by
``build.py`` with g++, loaded by ``stage.py``): FP32 elementwise steps with
the BF16 rounding points the pages name, exact sums of squares rounded once
to FP32, and a double-accumulated QKV dot product rounded once to FP32.
``preattn.py`` restates the same steps in PyTorch CPU ops; every pin runs on
both and the two agree bit for bit.  The neighbouring operations (output
projection, MLP block, e4m3 and NVFP4 outputs) are PyTorch CPU restatements
that call the C++ steps they share with the stage.

Pins: every function is pinned by tests that do not re-type its formula
(closed forms, library routines for special cases, exact integer arithmetic,
invariants, and a float64 brute-force recomputation of the whole stage on
tiny inputs).  No function here is "parity unpinned".
"""
from .stage import (  # noqa: F401
    input_rmsnorm,
    rmsnorm_apply,
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
from . import preattn  # noqa: F401  (PyTorch restatement of the same steps)
from . import out_proj  # noqa: F401  (attention output projection + gated residual)
from . import mlp  # noqa: F401  (MLP block)
from . import mlp_fp8  # noqa: F401  (FP8 MLP block)
from . import e4m3  # noqa: F401  (e4m3 output mode)
from . import nvfp4  # noqa: F401  (NVFP4 pre-attention)
