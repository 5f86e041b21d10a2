"""SageAttention2-style quantised non-causal attention for GB300 (sm_103a).

The compute path is the C-ABI CUDA library `_build/libsage_gb300.so` (include/sage.h);
this package is its thin Python binding (`_lib`) plus the seeded synthetic inputs
(`synth`).  Build with `build.build()`.
"""
from ._lib import (SageError, Quantized, dense_workspace, header_functions, lib, make_view, pad128, quant_scratch,
                   sage_attn_dense_bf16, sage_attn_dense_bf16_tc, sage_attn_fwd, sage_attn_fwd_quantized,
                   sage_check_device_status, sage_debug_qk_int32, sage_debug_wait_timeout, sage_measure_mma_rate,
                   sage_qk_rmsnorm_rope, sage_quant_qkv, sage_quant_v, sage_smooth_quant_qk,
                   sage_smooth_quant_qk_rmsnorm_rope, status_block, workspace)

__all__ = ["SageError", "Quantized", "dense_workspace", "header_functions", "lib", "make_view", "pad128",
           "quant_scratch", "sage_attn_dense_bf16", "sage_attn_dense_bf16_tc", "sage_attn_fwd",
           "sage_attn_fwd_quantized", "sage_check_device_status", "sage_debug_qk_int32", "sage_debug_wait_timeout",
           "sage_measure_mma_rate", "sage_qk_rmsnorm_rope", "sage_quant_qkv", "sage_quant_v", "sage_smooth_quant_qk",
           "sage_smooth_quant_qk_rmsnorm_rope", "status_block", "workspace"]
