"""Submanifold sparse convolution on one GB300 (sm_103a).

The compute path is libsc.so (CUDA, C ABI in include/sc.h); ``binding``
wraps it for torch tensors.  ``scenes`` draws seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    Hash,
    KernelMap,
    ScError,
    launch_count,
    lib,
    profile_collect,
    profile_enable,
    profile_only,
    profile_reset,
    sc_hash_build,
    sc_hash_build_conv_out,
    sc_kmap_build,
    sc_kmap_build_conv,
    sc_subm_conv_bwd_data,
    sc_subm_conv_bwd_weight,
    sc_subm_conv_fwd,
    sc_subm_conv_tune,
)
