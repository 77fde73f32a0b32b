"""GB300-native speculative-decoding verify-and-accept (libspecverify).

The compute path is the CUDA shared library built from ``csrc/`` (C ABI in
``include/spec_verify.h``); this package is its Python binding.  Names match
the C entry points: ``spec_verify_greedy``, ``spec_verify_sample``,
``spec_verify_workspace_bytes``, ``spec_verify_status`` …
"""
from .binding import (  # noqa: F401
    EXPORTED,
    MAX_GAMMA,
    SPEC_BF16,
    SPEC_ERR_ALIGNMENT,
    SPEC_ERR_CUDA,
    SPEC_ERR_DEVICE_INPUT,
    SPEC_ERR_INVALID_ARG,
    SPEC_ERR_TIMEOUT,
    SPEC_ERR_UNSUPPORTED,
    SPEC_ERR_STATE,
    SPEC_ERR_WORKSPACE,
    SPEC_F32,
    SPEC_OK,
    SpecRoundState,
    SpecVerifyError,
    error_string,
    lib_path,
    load,
    make_topkp_workspace,
    make_workspace,
    spec_round_update,
    spec_verify_greedy,
    spec_verify_greedy_multi,
    spec_verify_lmhead_gemm_only,
    spec_verify_lmhead_sample,
    spec_verify_sample,
    spec_verify_sample_noalloc,
    spec_verify_sample_topkp,
    spec_verify_sample_reduce_only,
    spec_verify_selftest_timeout,
    spec_verify_status,
    spec_verify_version,
    spec_verify_topkp_workspace_bytes,
    spec_verify_workspace_bytes,
    spec_verify_workspace_init,
)
