"""GB300 (sm_103a) hot path of batched Whisper large-v3 encoding.

libwb (CUDA, C ABI in include/wb.h) computes log-mel, the conv stem and the
encoder layers on the tensor cores; this package builds it and binds it.
"""
from ._lib import WB_BF16, WB_E4M3, WbError, load  # noqa: F401
from .api import (  # noqa: F401
    PRESET_AGGRESSIVE_FP8, PRESET_BF16, PRESET_MIXED_FP8, EncoderWeights, LayerWeights, Pipeline, StemWeights, attention,
    check_device_error, conv_stem, cross_kv, dequantize_e5m2, dequantize_fp8, encoder_forward, encoder_workspace_bytes,
    fold_layernorm, layernorm, layernorm_e4m3, linear,
    logmel, logmel_static, logmel_workspace_bytes, pack_conv_weight, profile_begin, profile_end, quantize_e5m2, quantize_fp8, rmsnorm, selftest_wait_timeout,
    upload_weights)
