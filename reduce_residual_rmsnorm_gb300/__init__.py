"""GB300 (sm_103a) fused "reduce R partials -> add residual -> RMSNorm ->
optional FP8 / NVFP4 quantise" epilogue and sharded MiniMax QK-RMSNorm.

The computation runs in ``libts_fused_norm.so`` (hand-written CUDA, C ABI in
include/ts_fused_norm.h); this package is its thin Python binding plus the
seeded synthetic workloads (``workloads``).  The library is loaded lazily, on
the first call.
"""
from ._binding import (EXPORTS, TS_FLAG_PDL, AGPattern, Pattern, RSPattern, SFLayout, TsError,  # noqa: F401
                       TsOuts, library, new_outputs, rs_token_split, sf_shape, sf_swizzled_shape,
                       ts_allgather_fused_norm, ts_fused_reduce_norm, ts_qk_norm_sharded,
                       ts_reducescatter_fused_norm, ts_rms_norm_sharded, ts_status_string)
