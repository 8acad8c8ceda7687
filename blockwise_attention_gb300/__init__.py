"""Blockwise multi-head attention with the Ring-Attention LSE merge, native to
NVIDIA GB300 (sm_103a).

The computation lives in libblockattn.so (C ABI in include/blockattn.h); the
functions here are its thin Python binding and allocate outputs with torch.
"""
from ._lib import (  # noqa: F401
    BA_BF16, BA_F32, BA_TILE_EMPTY, BA_TILE_FULL, BA_TILE_PARTIAL, BlockAttnError, EXPORTED, LIB_PATH,
    attn_block_bwd, attn_block_fwd, attn_decode_fwd, attn_block_fwd_noalloc, attn_merge, build, debug_wait_timeout, index_maps, load,
    pair_schedule, ring_attn_bwd, ring_attn_fwd, ring_attn_fwd_workspace_size, rope_apply, sync_status, tile_classes,
    ulysses_all_to_all, ulysses_attn_fwd,
)
