"""fp64 CPU oracle of the PowerSGD step (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
leg may import or execute anything here. The CUDA library neither imports this package
nor shares code with it. The product path fails loudly when its CUDA extension is
missing and never falls back to this code.
"""
from .numerics import (FORMATS, decode_bits, is_representable, max_finite, min_normal,
                       min_subnormal, round_to_format)
from .powersgd import (BlockResult, BlockState, PowerStepResult, accumulate_error,
                       block_step, compressed_fraction, error_update, orthonormalize,
                       power_step, scale_update, skip_block, skip_threshold,
                       uncompressed_mean, unscale_and_mask)

__all__ = [
    "FORMATS", "decode_bits", "is_representable", "max_finite", "min_normal",
    "min_subnormal", "round_to_format", "BlockResult", "BlockState", "PowerStepResult",
    "accumulate_error", "block_step", "compressed_fraction", "error_update",
    "orthonormalize", "power_step", "scale_update", "skip_block", "skip_threshold",
    "uncompressed_mean", "unscale_and_mask",
]
