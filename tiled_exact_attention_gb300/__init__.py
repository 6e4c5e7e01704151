"""GB300-native tiled exact attention (FlashAttention forward + split-KV decode).

The computation runs in libfa.so (hand-written sm_103a CUDA); this package only
marshals torch tensors into the C ABI of include/fa.h.
"""
from .api import (  # noqa: F401
    fa_bwd,
    fa_bwd_workspace_size,
    fa_fwd,
    fa_fwd_kvcache,
    fa_fwd_splitkv,
    fa_fwd_e4m3,
    fa_fwd_splitkv_noalloc,
    fa_fwd_splitkv_e4m3,
    fa_fwd_varlen,
    fa_num_splits_heuristic,
    fa_quantize_e4m3,
    quantize_qkv_e4m3,
    fa_selftest_wait_timeout,
    fa_splitkv_combine,
    fa_splitkv_default_splits,
    fa_splitkv_workspace_size,
    fa_sync_status,
    fa_version,
)
from ._lib import FaError  # noqa: F401
