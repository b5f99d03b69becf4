"""combine_ep_layout_gb300 -- single-GPU MoE expert-parallel layout, dispatch
and combine for GB300 (sm_103a): a C-ABI CUDA library (libep_gb300.so) and its
thin Python binding.  See include/ep_gb300.h for the contract of each call."""
from ._native import (  # noqa: F401
    EP_BF16, EP_FP32, EP_FP8_E4M3, EP_FP4X2,
    EP_OK, EP_EINVAL, EP_EUNSUPPORTED, EP_ECUDA, EP_ENOMEM,
    FIELD_NUM_UNALIGNED_PER_EXPERT, FIELD_NUM_TOKENS_PER_RANK, FIELD_PSUM_PER_EXPERT,
    FIELD_PSUM_PER_RANK, FIELD_DST_SLOT, FIELD_RECV_SRC_METADATA, FIELD_NUM_RECV,
    FIELD_DEVICE_ERROR, FIELD_TOPK_IDX, FIELD_SEND_SLOT, ERR_BAD_EXPERT, ERR_TIMEOUT,
    EpError, EpHandle, ep_cfg_t, make_cfg, load_library, declared_symbols,
    ep_recv_capacity, ep_handle_create, ep_handle_create_shared, ep_layout, ep_dispatch, ep_combine, ep_handle_free,
    ep_handle_get, ep_handle_status, ep_handle_variant, ep_last_error,
    ep_layout_noalloc, NOALLOC_OUTPUTS, ep_dispatch_fwd, ep_combine_ex, ep_jit_precompile,
)
