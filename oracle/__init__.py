"""Independent float64 CPU oracle of the Muon step (test infrastructure).

Only tests, the package smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never does.
"""
from .muon_ref import (  # noqa: F401
    column_blocks,
    frobenius_normalise,
    momentum_update,
    muon_step,
    muon_step_matrix,
    newton_schulz,
    newton_schulz_distributed,
    shape_scale,
    shard_ranges,
)
