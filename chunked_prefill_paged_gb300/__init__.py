"""GB300-native (sm_103a) paged chunked-prefill attention.

A mixed batch of active tokens -- prefill chunks under a per-step token
budget plus single-token decodes -- attends to each request's block-paged
K/V cache and, causally, to its own chunk; the new K/V rows are written into
their pool slots.  The computation lives in libcpa.so (C ABI in
include/cpa.h); this package is its ctypes binding.
"""
from .binding import (  # noqa: F401
    DTYPE_BF16,
    DTYPE_FP32,
    ERR_BAD_BLOCK_ID,
    ERR_CUDA,
    ERR_DEVICE_TIMEOUT,
    ERR_INVALID_ARG,
    ERR_UNSUPPORTED,
    ERR_WORKSPACE,
    EXPORTED,
    FLAG_FORCE_SIMT,
    FLAG_FUSE_KV_WRITE,
    FLAG_NO_SPLIT,
    FLAG_TAIL_SPLIT,
    FLAG_TEST_STALL,
    KV_FP8_E4M3,
    KV_SAME,
    LIB_PATH,
    NO_ALLOC_WORKSPACE_BYTES,
    SUCCESS,
    Batch,
    CpaError,
    Engine,
    StepPlan,
    Params,
    attention,
    chunked_prefill_attention,
    chunked_prefill_attention_no_alloc,
    last_device_error,
    load,
    paged_kv_write,
    status_string,
    workspace_size,
)
