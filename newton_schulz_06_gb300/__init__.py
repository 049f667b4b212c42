"""libmuon for GB300: the Muon optimizer step (momentum, Frobenius
normalisation, quintic Newton-Schulz orthogonalisation with tcgen05
tensor-core kernels, shape-scaled update) over many matrices at once.

The compute lives in the C-ABI shared library libmuon.so (include/muon.h);
this package only binds it.  Build with ``python -m
newton_schulz_06_gb300.build``.
"""
from ._lib import (MUON_BF16, MUON_BLOCKWISE, MUON_DISTRIBUTED,  # noqa
                   MUON_F32, MUON_FULL, MuonError)
from .flops import gemm_equiv_flops, useful_flops  # noqa: F401
from .muon import DEFAULT_COEFFS, HostPlanner, Muon, mode_code  # noqa: F401
from .layerwise import LayerwiseMuon, lpt_partition  # noqa: F401
