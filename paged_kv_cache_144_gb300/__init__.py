"""GB300 (sm_103a) paged decode attention: decode, cache write and CoW block copy.

The compute path is libpagedattn.so (hand-written CUDA kernels behind the C ABI
in include/pa.h); this package holds its build script, the ctypes binding and
the host-side block manager.
"""

from ._lib import (  # noqa: F401
    PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3, PA_INT8,
    PA_OK, PA_ERR_NULL, PA_ERR_SHAPE, PA_ERR_DTYPE, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA,
    PA_ERR_ALIGN, PA_DEVERR_BLOCK_ID, PA_DEVERR_SLOT, PA_DEVERR_SEQ_LEN, PA_DEVERR_TIMEOUT, PA_DEVERR_PAIR,
    PagedAttnError, load, header_functions, status_string,
    pa_decode, pa_decode_ex, DecodeOptions, CacheWriteOptions, pa_reshape_and_cache, pa_reshape_and_cache_ex,
    pa_copy_blocks, pa_decode_workspace_bytes,
    pa_get_device_error,
    pa_version, pa_decode_launch_config, pa_decode_noalloc, pa_decode_noalloc_capacity, decode_noalloc,
    pa_debug_set_decode_wait,
    decode, reshape_and_cache, copy_blocks, decode_workspace_bytes, new_workspace, get_device_error,
    dtype_code,
)
from .block_manager import BlockManager  # noqa: F401
from .step_graph import StepGraph  # noqa: F401
