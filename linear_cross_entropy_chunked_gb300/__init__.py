"""GB300 (sm_103a) fused chunked linear + cross-entropy.

The compute runs in liblce_gb300.so (tcgen05/TMEM/TMA kernels behind a C ABI,
include/lce.h); this package is the thin ctypes binding around it.
"""
from ._binding import (  # noqa: F401
    ACCUMULATE,
    EXPORTED,
    FROZEN_W,
    IGNORE_INDEX,
    INPUT_FP16,
    KERNEL_KINDS,
    LCEError,
    LOW_MEMORY,
    LinearCrossEntropyFunction,
    NormLinearCrossEntropyFunction,
    alloc_workspace,
    ce_logits,
    count_valid,
    forward_noalloc,
    forward_workspace_size,
    last_launch_count,
    lce_backward,
    lce_forward,
    lce_fwd_bwd,
    lib,
    linear_cross_entropy,
    norm_fwd_bwd,
    norm_linear_cross_entropy,
    noalloc_read_status,
    norm_workspace_size,
    profile_enable,
    profile_read,
    profile_reset,
    read_status,
    rmsnorm_backward,
    rmsnorm_forward,
    selftest_wait_timeout,
    workspace_size,
    workspace_size_opt,
)
from .build_lib import LIB_PATH, build  # noqa: F401
from .sharded import sharded_fwd_bwd  # noqa: F401
