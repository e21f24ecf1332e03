"""GB300-native (sm_103a) KDA RecoverSSM step for speculative decoding.

The compute lives in libkda_recoverssm.so (hand-written CUDA kernels behind a
C ABI, declared in include/kda_recoverssm.h).  This package holds the build
script (``_build``), the thin ctypes binding (``_lib``), the deferred
RecoverSSM's step sequencing across decode steps (``decode``) and the seeded
synthetic-input generator (``synth``).  Calling any entry point without the
built library raises ImportError; there is no CPU fallback.
"""
from ._lib import (  # noqa: F401
    EXPORTS,
    KDA_ERR_ALIGN,
    KDA_ERR_ARG,
    KDA_ERR_CUDA,
    KDA_ERR_SCRATCH,
    KDA_ERR_TIMEOUT,
    KDA_ERR_UNSUPPORTED,
    KDA_LAYER_STEP_NOALLOC_MAX_BYTES,
    KDA_OK,
    KDA_STATE_BF16,
    KDA_STATE_F32,
    KdaError,
    kda_check_status,
    kda_commit,
    kda_defer_commit,
    kda_flush_plan,
    kda_layer_epilogue,
    kda_layer_prologue,
    kda_layer_step,
    kda_layer_step_noalloc,
    kda_layer_step_workspace_bytes,
    kda_replay_verify,
    kda_replay_verify_layers,
    kda_selftest_wait_timeout,
    kda_verify,
    layer_tables,
    load,
)
from .decode import DeferredRecoverSSM  # noqa: F401
