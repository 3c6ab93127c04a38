"""Float64 CPU oracle for the FLASH GAU forward (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and the
two share no code.
"""

from .flash_gau import (  # noqa: F401
    swish,
    scale_offset,
    relpos_bias,
    chunk_scores,
    chunk_mask,
    layer_norm,
    scale_norm,
    rope,
    rope_toeplitz_bias,
    toeplitz_relpos,
    flash_gau,
    flash_block,
    algorithmic_flops_per_token,
)
from .backward import swish_grad, flash_gau_backward  # noqa: F401,E402
from .decode import DecodeState  # noqa: F401,E402
