"""GB300-native (sm_103a) TwELL activation-sparse feed-forward layer.

The compute path is the CUDA library ``libtwell.so`` (C ABI in
``include/twell.h``); ``twell`` is its thin ctypes binding (argument
marshalling only). Nothing here computes on the CPU.
"""
from .twell import (TwellBuffers, TwellOverflow, TwellError, load_library, twell_buf_slots_bound, twell_check,
                    twell_dense_ffn_fwd, twell_dense_ffn_bwd, twell_dense_bwd_workspace_bytes,
                    twell_device_sm_count, twell_ffn_bwd, twell_ffn_fwd, twell_pack,
                    twell_spmm_down, twell_status_string, twell_workspace_bytes, twell_fwd_workspace_bytes, twell_up_pack,
                    twell_kernel_launches, twell_ffn_fwd_static_ws, twell_set_kernel_timer, twell_hybrid_up_pack, twell_hybrid_spmm_down, twell_hybrid_ffn_fwd,
                    twell_hybrid_ffn_bwd, twell_hybrid_bwd_workspace_bytes, twell_wait_selftest, twell_spmm_down_tc,
                    twell_spmm_down_tc_workspace_bytes, STATIC_WS_BYTES, OP_PACK, OP_SPMM_DOWN, OP_HYBRID_FWD,
                    OP_FFN_FWD, OP_FFN_BWD, OP_GATED_FWD, EXPORTED_SYMBOLS)

__all__ = [
    "TwellBuffers", "TwellOverflow", "TwellError", "load_library", "twell_buf_slots_bound", "twell_check",
    "twell_dense_ffn_fwd", "twell_dense_ffn_bwd", "twell_dense_bwd_workspace_bytes", "twell_device_sm_count", "twell_ffn_bwd", "twell_ffn_fwd", "twell_pack",
    "twell_spmm_down", "twell_status_string", "twell_workspace_bytes", "twell_fwd_workspace_bytes", "twell_up_pack",
    "twell_kernel_launches", "twell_ffn_fwd_static_ws", "twell_set_kernel_timer", "twell_hybrid_up_pack", "twell_hybrid_spmm_down", "twell_hybrid_ffn_fwd",
    "twell_hybrid_ffn_bwd", "twell_hybrid_bwd_workspace_bytes", "twell_wait_selftest", "twell_spmm_down_tc",
    "twell_spmm_down_tc_workspace_bytes", "STATIC_WS_BYTES", "OP_PACK", "OP_SPMM_DOWN", "OP_HYBRID_FWD",
    "OP_FFN_FWD", "OP_FFN_BWD", "OP_GATED_FWD", "EXPORTED_SYMBOLS",
]
