"""GB300 (sm_103a) paged Multi-head Latent Attention decode.

The compute path is the C-ABI shared library declared in include/mla_decode.h
(hand-written tcgen05/TMA kernels). This package is its thin Python binding;
PyTorch supplies device memory and streams only.
"""
from ._lib import (MLAError, Plan, mla_check_device_error, mla_decode, mla_decode_plan,  # noqa: F401
                   mla_device_supported, mla_status_string, header_functions,
                   MLA_DEVERR_BAD_BLOCK, MLA_DEVERR_SEQLEN_MISMATCH, MLA_DEVERR_TIMEOUT)
from .api import decode  # noqa: F401
