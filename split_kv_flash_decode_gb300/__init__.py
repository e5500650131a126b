"""GB300-native split-KV Flash Decode.

One query token per sequence attends over a long KV cache split into W
segments; per-segment partials (O, m, l) are merged by OnlineSoftmaxCombine
inside the same kernel by the last-arriving CTA.  The compute lives in
``csrc/`` (hand-written sm_103a CUDA behind the C ABI of ``include/fd.h``);
this package is its thin Python binding plus a convenience wrapper that
allocates outputs and workspace with PyTorch.
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    FD_BF16,
    FD_ERR_ALIGN,
    FD_ERR_CUDA,
    FD_ERR_INVALID,
    FD_ERR_NOMEM,
    FD_ERR_STATE,
    FD_ERR_TIMEOUT,
    FD_ERR_UNSUPPORTED,
    FD_F16,
    FD_F16_E4M3KV,
    FD_MAX_BATCH,
    FD_MAX_PARTIALS,
    FD_NOALLOC_SCRATCH_BYTES,
    FD_OK,
    FD_PLAN_DEBUG,
    FD_PLAN_FFMA,
    FD_PLAN_LITERAL_W,
    FD_PLAN_CLUSTER,
    FD_PLAN_NO_CLUSTER,
    FD_PLAN_NO_PDL,
    FD_PLAN_TEST_DROP_FLAG,
    FD_PLAN_TEST_SKIP_TILE,
    FD_PLAN_TEST_DROP_ARRIVAL,
    FD_PLAN_DEEP_RING,
    FD_PLAN_TCGEN05,
    FD_PLAN_CLUSTER_COMBINE,
    FD_PLAN_MMA_SYNC,
    FD_PLAN_SINGLE_COMBINER,
    FD_PLAN_COMBINERS,
    FD_PLAN_COMBINERS_MASK,
    FD_PLAN_WAITS,
    FD_PLAN_TWO_LAUNCH,
    FdError,
    Plan,
    fd_decode,
    fd_decode_noalloc,
    fd_noalloc_status,
    fd_decode_paged,
    fd_plan,
    fd_plan_paged,
    fd_plan_destroy,
    fd_plan_get_range,
    fd_version,
    fd_workspace_bytes,
    fd_workspace_init,
    fd_workspace_status,
    lib,
    strerror as fd_strerror,
)
from .decode import Decoder, flash_decode  # noqa: F401
