"""GB300 (sm_103a) forward pass of the FLASH gated attention unit with mixed
chunk attention ("Transformer Quality in Linear Time").

The computation lives in libflashgau.so (C ABI in include/flash_gau.h); this
package holds its build step, a ctypes binding and the seeded synthetic
input generator used by the tests and the benchmark.
"""

from .binding import (  # noqa: F401
    FP32, BF16, GauWeights, FlashGauError, forward, workspace_layout,
    workspace_status, num_stages, stage_names, lib, strerror, EXPORTED,
)

__version__ = "0.1.0"
