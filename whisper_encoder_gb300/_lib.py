"""ctypes binding of libwb (include/wb.h): argument marshalling only.

Every step of the hot path runs in libwb's CUDA kernels; torch is used here
for device memory (tensor allocation) and for the current CUDA stream.  If the
library has not been built, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

LIB_PATH = _build.LIB

WB_OK, WB_EINVAL, WB_ECUDA, WB_EUNSUPPORTED, WB_ETIMEOUT, WB_EWORKSPACE, WB_EBOUNDS = 0, -1, -2, -3, -4, -5, -6
WB_BF16, WB_E4M3 = 0, 1
WB_LOGMEL_STATIC_MAX_CHUNKS = 2   # include/wb.h
WB_SELFTEST_WAIT_SITE = 0x7F      # include/wb.h
WB_SELFTEST_BOUNDS_SITE = 0x7E    # include/wb.h

c_int, c_i64, c_size, c_void, c_float = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
P = ctypes.POINTER


class wb_precision(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("qkv_w", "qkv_a", "out_w", "out_a", "ffn_w", "ffn_a")]


class wb_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_mels", "d_model", "n_heads", "n_layers", "d_ffn")]


class wb_stem_weights(ctypes.Structure):
    _fields_ = [("conv1_w", c_void), ("conv1_b", c_void), ("conv2_w", c_void), ("conv2_b", c_void)]


class wb_layer_weights(ctypes.Structure):
    _fields_ = [(n, c_void) for n in (
        "ln1_g", "ln1_b", "w_qkv", "b_qkv", "s_qkv", "w_out", "b_out", "s_out", "ln2_g", "ln2_b",
        "w_fc1", "b_fc1", "s_fc1", "w_fc2", "b_fc2", "s_fc2",
        "w_qkv_ln", "c_qkv", "b_qkv_ln", "w_fc1_ln", "c_fc1", "b_fc1_ln")]


class wb_cross_kv_weights(ctypes.Structure):
    _fields_ = [("w_kv", c_void), ("b_kv", c_void)]


class wb_ln_weights(ctypes.Structure):
    _fields_ = [("g", c_void), ("b", c_void)]


class wb_host_pipeline(ctypes.Structure):
    _fields_ = [("dims", wb_dims), ("batch", ctypes.c_int32), ("samples_per_batch", ctypes.c_int64),
                ("chunk_stride", ctypes.c_int64), ("stem", P(wb_stem_weights)), ("layers", P(wb_layer_weights)),
                ("ln_post", P(wb_ln_weights)), ("precision", wb_precision), ("dev_audio", c_void * 2),
                ("dev_mel", c_void), ("dev_x0", c_void), ("dev_out", c_void * 2), ("ws_mel", c_void),
                ("ws_mel_bytes", c_size), ("ws_stem", c_void), ("ws_stem_bytes", c_size), ("ws_enc", c_void),
                ("ws_enc_bytes", c_size), ("upload_stream", c_void), ("download_stream", c_void)]


# name -> (restype, argtypes); must match include/wb.h
SIGNATURES = {
    "wb_status_string": (ctypes.c_char_p, [c_int]),
    "wb_version": (c_int, []),
    "wb_debug_build": (c_int, []),
    "wb_check_device_error": (c_int, [c_void, P(ctypes.c_uint32)]),
    "wb_selftest_wait_timeout": (c_int, [c_void]),
    "wb_selftest_bounds_check": (c_int, [c_void]),
    "wb_logmel_workspace_bytes": (c_size, [c_int, c_int]),
    "wb_logmel": (c_int, [c_void, c_i64, c_i64, c_int, c_int, c_void, c_void, c_size, c_void]),
    "wb_logmel_static": (c_int, [c_void, c_i64, c_i64, c_int, c_int, c_void, c_void]),
    "wb_conv_stem_workspace_bytes": (c_size, [P(wb_dims), c_int]),
    "wb_conv_stem": (c_int, [c_void, c_int, P(wb_dims), P(wb_stem_weights), c_void, c_void, c_size, c_void]),
    "wb_pack_conv_weight": (c_int, [c_void, c_int, c_int, c_void, c_void]),
    "wb_encoder_workspace_bytes": (c_size, [P(wb_dims), c_int, P(wb_precision)]),
    "wb_encoder_forward": (c_int, [c_void, c_int, P(wb_dims), P(wb_layer_weights), P(wb_ln_weights),
                                   P(wb_precision), c_int, c_int, c_int, c_void, c_void, c_size, c_void]),
    "wb_encode_host": (c_int, [P(wb_host_pipeline), P(c_void), P(c_void), c_int, c_void]),
    "wb_quantize_fp8": (c_int, [c_void, c_i64, c_void, c_void, c_void]),
    "wb_fold_layernorm": (c_int, [c_void, c_void, c_void, c_void, c_int, c_int, c_void, c_void, c_void, c_void]),
    "wb_dequantize_fp8": (c_int, [c_void, c_void, c_i64, c_void, c_void]),
    "wb_linear": (c_int, [c_void, c_void, c_int, c_int, c_int, c_int, c_void, c_void, c_void, c_int, c_void,
                          c_void, c_void]),
    "wb_layernorm": (c_int, [c_void, c_void, c_void, c_void, c_int, c_int, c_float, c_void, c_void, c_void]),
    "wb_layernorm_e4m3": (c_int, [c_void, c_void, c_void, c_int, c_int, c_float, c_int, c_void, c_void, c_void,
                                  c_void]),
    "wb_attention_workspace_bytes": (c_size, [c_int, c_int, c_int]),
    "wb_attention": (c_int, [c_void, c_void, c_void, c_int, c_int, c_int, c_void, c_void, c_size, c_void]),
    "wb_cross_kv": (c_int, [c_void, c_int, P(wb_dims), c_int, P(wb_cross_kv_weights), c_void, c_void]),
    "wb_rmsnorm": (c_int, [c_void, c_void, c_void, c_int, c_int, c_float, c_void, c_void, c_void]),
    "wb_quantize_e5m2": (c_int, [c_void, c_i64, c_void, c_void, c_void]),
    "wb_dequantize_e5m2": (c_int, [c_void, c_void, c_i64, c_void, c_void]),
    "wb_profile_begin": (c_int, []),
    "wb_profile_end": (c_int, [c_int, P(ctypes.c_char_p), P(ctypes.c_double), P(ctypes.c_int64)]),
}

_LIB = None


class WbError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = status_string(status) if _LIB is not None else str(status)
        super().__init__(f"{fn} failed: {msg} ({status})")


def open_library(path: str) -> ctypes.CDLL:
    """Open a build of libwb at ``path`` with the ctypes signatures of include/wb.h."""
    if not os.path.exists(path):
        raise RuntimeError(f"libwb is not built ({path}); run `python -m whisper_encoder_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libwb.so (built beforehand by whisper_encoder_gb300.build)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    _LIB = open_library(path or LIB_PATH)
    return _LIB


def status_string(status: int) -> str:
    return load().wb_status_string(status).decode()


def call(name: str, *args) -> None:
    st = getattr(load(), name)(*args)
    if st != WB_OK:
        raise WbError(name, st)
