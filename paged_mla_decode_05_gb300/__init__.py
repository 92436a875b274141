"""GB300 (sm_103a) paged Multi-head Latent Attention decode.

The compute path is the C-ABI shared library declared in include/mla_decode.h
(hand-written tcgen05/TMA kernels). This package is its thin Python binding;
PyTorch supplies device memory and streams only.

The binding loads the library on first use of any exported name; if the
library has not been built (``python -m paged_mla_decode_05_gb300.build``)
that first use raises ImportError. There is no fallback path.
"""
_EXPORTS = ("MLAError", "Plan", "mla_check_device_error", "mla_decode", "mla_decode_fp8",
            "mla_decode_no_alloc", "mla_sparse_plan", "mla_decode_sparse",
            "mla_decode_plan",
            "mla_device_supported", "mla_selftest_wait_timeout", "mla_status_string",
            "header_functions",
            "MLA_DEVERR_BAD_BLOCK", "MLA_DEVERR_SEQLEN_MISMATCH", "MLA_DEVERR_TIMEOUT")


def __getattr__(name):
    if name in _EXPORTS:
        from . import _lib
        return getattr(_lib, name)
    if name in ("decode", "decode_sparse"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)


__all__ = list(_EXPORTS) + ["decode", "decode_sparse"]
