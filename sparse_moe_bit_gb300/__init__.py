"""Sparse 4-bit Mixture-of-Experts block for GB300 (sm_103a).

The compute lives in libmoe.so (CUDA kernels behind the C ABI of
include/moe.h, and the Gated DeltaNet prefill scan of include/gdn.h); this
package is its thin Python binding.
"""
from .moe import (MOE_DEVERR_FP16_RANGE, MOE_DEVERR_GRID_TIMEOUT, MOE_DEVERR_NAN_LOGIT,
                  MOE_DEVERR_RANGE, MOE_DEVERR_WAIT_TIMEOUT, MOE_LAYOUT_DECODE,
                  MOE_LAYOUT_PREFILL, MOE_SCALE_F16, MoE, MoEConfig, MoEError, decode,
                  decode_host, gdn_scan, load_library)

__all__ = ["MoE", "MoEConfig", "MoEError", "decode", "decode_host", "gdn_scan", "load_library",
           "MOE_SCALE_F16", "MOE_LAYOUT_PREFILL", "MOE_LAYOUT_DECODE", "MOE_DEVERR_WAIT_TIMEOUT",
           "MOE_DEVERR_NAN_LOGIT", "MOE_DEVERR_GRID_TIMEOUT", "MOE_DEVERR_RANGE",
           "MOE_DEVERR_FP16_RANGE"]
