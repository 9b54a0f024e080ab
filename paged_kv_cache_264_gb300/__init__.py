"""GB300 (sm_103a) PagedAttention decode: a C-ABI library of hand-written CUDA kernels
(``include/pagedkv.h``, sources in ``csrc/``) and this thin Python binding.

The library is loaded on first use; importing the package does not need a GPU.
"""

from .api import (  # noqa: F401
    BlockManager,
    PagedKVPool,
    copy_blocks,
    decode_plan,
    decode_workspace_bytes,
    get_device_error,
    launch_count,
    paged_attention_decode,
    pool_bytes,
    pool_create,
    pool_destroy,
    reshape_and_cache,
    selftest_bounded_wait,
    version,
)
from ._lib import (  # noqa: F401
    BLOCK_SIZE,
    DEVERR_BLOCK_ID,
    DEVERR_CONTEXT_LEN,
    DEVERR_SLOT,
    DEVERR_TIMEOUT,
    PagedKVError,
)
