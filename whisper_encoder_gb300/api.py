"""Python surface of libwb: one function per C entry point, plus weight upload.

Argument marshalling only: tensors are checked for device, dtype and
contiguity, workspaces are allocated with torch, and the C call runs on the
current torch CUDA stream.  All arithmetic happens in libwb's kernels.
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _lib
from ._lib import WB_BF16, WB_E4M3, WB_ETIMEOUT, WB_OK, WbError, call, load

CHUNK_SAMPLES = 480000
N_FRAMES = 3000
N_TOKENS = 1500

PRESET_BF16 = (WB_BF16,) * 6
PRESET_MIXED_FP8 = (WB_E4M3, WB_E4M3, WB_BF16, WB_BF16, WB_E4M3, WB_E4M3)   # qkv, out, ffn (w, a)
PRESET_AGGRESSIVE_FP8 = (WB_E4M3,) * 6                                        # every encoder site in E4M3


def _p(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor")


def _need_out(t, dtype, shape, device, name):
    """A caller-supplied output must be exactly what the kernel writes: the kernels write every
    element of the given shape and nothing is checked on the device."""
    _need(t, dtype, name)
    if tuple(t.shape) != tuple(shape) or t.device != device:
        raise ValueError(f"{name}: expected shape {tuple(shape)} on {device}, got {tuple(t.shape)} on {t.device}")


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def dims_struct(d) -> _lib.wb_dims:
    return _lib.wb_dims(d.n_mels, d.d_model, d.n_heads, d.n_layers, d.d_ffn)


def precision_struct(p) -> _lib.wb_precision:
    return _lib.wb_precision(*p)


# ------------------------------- log-mel -------------------------------------
def logmel_workspace_bytes(n_chunks: int, n_mels: int) -> int:
    return load().wb_logmel_workspace_bytes(n_chunks, n_mels)


def logmel(audio: torch.Tensor, n_chunks: int, n_mels: int, chunk_stride: int = CHUNK_SAMPLES,
           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """float32 audio (device, 1-D) -> float32 log-mel [n_chunks, n_mels, 3000]."""
    _need(audio, torch.float32, "audio")
    if out is None:
        out = torch.empty((n_chunks, n_mels, N_FRAMES), dtype=torch.float32, device=audio.device)
    _need_out(out, torch.float32, (n_chunks, n_mels, N_FRAMES), audio.device, "out")
    if workspace is None:
        workspace = _workspace(logmel_workspace_bytes(n_chunks, n_mels), audio.device)
    call("wb_logmel", _p(audio), audio.numel(), chunk_stride, n_chunks, n_mels, _p(out), _p(workspace),
         workspace.numel(), _stream(stream))
    return out


def logmel_static(audio: torch.Tensor, n_chunks: int, n_mels: int, chunk_stride: int = CHUNK_SAMPLES,
                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """wb_logmel without a workspace: scratch comes from the library's fixed device array.

    For callers that must not allocate device memory; at most
    WB_LOGMEL_STATIC_MAX_CHUNKS chunks per call, and calls must not overlap on the GPU.
    (``out`` is allocated here only when the caller passes none.)"""
    _need(audio, torch.float32, "audio")
    if out is None:
        out = torch.empty((n_chunks, n_mels, N_FRAMES), dtype=torch.float32, device=audio.device)
    _need_out(out, torch.float32, (n_chunks, n_mels, N_FRAMES), audio.device, "out")
    call("wb_logmel_static", _p(audio), audio.numel(), chunk_stride, n_chunks, n_mels, _p(out), _stream(stream))
    return out


# ------------------------------- conv stem -----------------------------------
def pack_conv_weight(w: torch.Tensor, stream=None) -> torch.Tensor:
    """float32 [c_out, c_in, 3] (device) -> bf16 tap-major [3, c_out, c_in]."""
    _need(w, torch.float32, "w")
    c_out, c_in, k = w.shape
    assert k == 3
    packed = torch.empty((3, c_out, c_in), dtype=torch.bfloat16, device=w.device)
    call("wb_pack_conv_weight", _p(w), c_out, c_in, _p(packed), _stream(stream))
    return packed


def conv_stem(mel: torch.Tensor, dims, stem: "StemWeights", out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need(mel, torch.float32, "mel")
    batch = mel.shape[0]
    ds = dims_struct(dims)
    if out is None:
        out = torch.empty((batch, N_TOKENS, dims.d_model), dtype=torch.bfloat16, device=mel.device)
    _need_out(out, torch.bfloat16, (batch, N_TOKENS, dims.d_model), mel.device, "out")
    if workspace is None:
        workspace = _workspace(load().wb_conv_stem_workspace_bytes(ctypes.byref(ds), batch), mel.device)
    call("wb_conv_stem", _p(mel), batch, ctypes.byref(ds), ctypes.byref(stem.struct()), _p(out), _p(workspace),
         workspace.numel(), _stream(stream))
    return out


# -------------------------------- encoder ------------------------------------
def encoder_workspace_bytes(dims, batch: int, precision=PRESET_BF16) -> int:
    ds, pr = dims_struct(dims), precision_struct(precision)
    return load().wb_encoder_workspace_bytes(ctypes.byref(ds), batch, ctypes.byref(pr))


def encoder_forward(x0: torch.Tensor, dims, weights: "EncoderWeights", precision=PRESET_BF16,
                    layer_begin: int = 0, layer_end: int | None = None, final_ln: bool = True,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    _need(x0, torch.bfloat16, "x0")
    batch = x0.shape[0]
    if layer_end is None:
        layer_end = dims.n_layers
    ds, pr = dims_struct(dims), precision_struct(precision)
    if out is None:
        out = torch.empty_like(x0)
    _need_out(out, torch.bfloat16, tuple(x0.shape), x0.device, "out")
    if workspace is None:
        workspace = _workspace(encoder_workspace_bytes(dims, batch, precision), x0.device)
    layers = weights.layer_array(precision)
    ln = _lib.wb_ln_weights(weights.ln_post_g.data_ptr(), weights.ln_post_b.data_ptr())
    call("wb_encoder_forward", _p(x0), batch, ctypes.byref(ds), layers, ctypes.byref(ln), ctypes.byref(pr),
         layer_begin, layer_end, 1 if final_ln else 0, _p(out), _p(workspace), workspace.numel(), _stream(stream))
    return out


# ---------------------------------- FP8 ---------------------------------------
def quantize_fp8(x: torch.Tensor, stream=None):
    """bf16 tensor -> (uint8 E4M3 codes, float32 device scale [1])."""
    _need(x, torch.bfloat16, "x")
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scale = torch.empty(1, dtype=torch.float32, device=x.device)
    call("wb_quantize_fp8", _p(x), x.numel(), _p(q), _p(scale), _stream(stream))
    return q, scale


def fold_layernorm(w: torch.Tensor, b, gamma: torch.Tensor, beta: torch.Tensor, stream=None):
    """LayerNorm (gamma, beta) folded into the linear layer (w bf16 [n, d], b f32 [n] or None) after it:
    returns (w_ln bf16 [n, d], c f32 [n], b_ln f32 [n]) for wb_encoder_forward's folded sites."""
    _need(w, torch.bfloat16, "w")
    n, d = w.shape
    w_ln = torch.empty_like(w)
    c = torch.empty(n, dtype=torch.float32, device=w.device)
    b_ln = torch.empty(n, dtype=torch.float32, device=w.device)
    call("wb_fold_layernorm", _p(w), _p(b), _p(gamma), _p(beta), n, d, _p(w_ln), _p(c), _p(b_ln), _stream(stream))
    return w_ln, c, b_ln


def dequantize_fp8(q: torch.Tensor, scale: torch.Tensor, stream=None) -> torch.Tensor:
    _need(q, torch.uint8, "q")
    y = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    call("wb_dequantize_fp8", _p(q), _p(scale), q.numel(), _p(y), _stream(stream))
    return y


# ----------------------------- building blocks --------------------------------
def linear(a, w, bias=None, scale_a=None, scale_w=None, gelu=False, resid=None, stream=None) -> torch.Tensor:
    fp8 = a.dtype == torch.uint8
    _need(a, a.dtype, "a")
    _need(w, a.dtype, "w")
    M, K = a.shape
    N = w.shape[0]
    out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    call("wb_linear", _p(a), _p(w), M, N, K, WB_E4M3 if fp8 else WB_BF16, _p(bias), _p(scale_a), _p(scale_w),
         1 if gelu else 0, _p(resid), _p(out), _stream(stream))
    return out


def layernorm(x, g, b, eps: float = 1e-5, residual=None, return_total: bool = False, stream=None):
    _need(x, torch.bfloat16, "x")
    rows, d = x.reshape(-1, x.shape[-1]).shape
    y = torch.empty_like(x)
    total = torch.empty_like(x) if return_total else None
    call("wb_layernorm", _p(x), _p(residual), _p(g), _p(b), rows, d, eps, _p(y), _p(total), _stream(stream))
    return (y, total) if return_total else y


def layernorm_e4m3(x, g, b, eps: float = 1e-5, rows_per_item: int | None = None, stream=None):
    """LayerNorm to E4M3 codes with one absmax scale per item of rows_per_item rows (default: all rows).

    Returns (codes u8 [rows, d], amax f32 [items], stats f32 [rows, 2] = (mean, rstd)); the
    dequantised output is codes * amax[item] / 448."""
    _need(x, torch.bfloat16, "x")
    x2 = x.reshape(-1, x.shape[-1])
    rows, d = x2.shape
    rpi = rows if rows_per_item is None else int(rows_per_item)
    items = (rows + rpi - 1) // rpi if rows else 0
    q = torch.empty((rows, d), dtype=torch.uint8, device=x.device)
    amax = torch.empty(max(items, 1), dtype=torch.float32, device=x.device)
    stats = torch.empty((max(rows, 1), 2), dtype=torch.float32, device=x.device)
    call("wb_layernorm_e4m3", _p(x2), _p(g), _p(b), rows, d, eps, max(rpi, 1), _p(q), _p(amax), _p(stats),
         _stream(stream))
    return q, amax[:items], stats[:rows]


def attention(q, k, v, n_heads: int, stream=None) -> torch.Tensor:
    """q, k, v: bf16 [batch, T, 64*n_heads] -> softmax(q k^T / 8) v per head."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    batch, T, _ = q.shape
    out = torch.empty_like(q)
    ws = _workspace(load().wb_attention_workspace_bytes(batch, T, n_heads), q.device)
    call("wb_attention", _p(q), _p(k), _p(v), batch, T, n_heads, _p(out), _p(ws), ws.numel(), _stream(stream))
    return out


def rmsnorm(x, g, eps: float = 1e-5, residual=None, return_total: bool = False, stream=None):
    _need(x, torch.bfloat16, "x")
    rows, d = x.reshape(-1, x.shape[-1]).shape
    y = torch.empty_like(x)
    total = torch.empty_like(x) if return_total else None
    call("wb_rmsnorm", _p(x), _p(residual), _p(g), rows, d, eps, _p(y), _p(total), _stream(stream))
    return (y, total) if return_total else y


def quantize_e5m2(x: torch.Tensor, stream=None):
    _need(x, torch.bfloat16, "x")
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scale = torch.empty(1, dtype=torch.float32, device=x.device)
    call("wb_quantize_e5m2", _p(x), x.numel(), _p(q), _p(scale), _stream(stream))
    return q, scale


def dequantize_e5m2(q: torch.Tensor, scale: torch.Tensor, stream=None) -> torch.Tensor:
    _need(q, torch.uint8, "q")
    y = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    call("wb_dequantize_e5m2", _p(q), _p(scale), q.numel(), _p(y), _stream(stream))
    return y


def cross_kv(enc_out: torch.Tensor, dims, layers: list, stream=None) -> torch.Tensor:
    """Decoder cross-attention K|V of the encoder output for every decoder layer.

    layers: per decoder layer (w_kv bf16 [2d, d], b_kv f32 [2d]); returns bf16 [L, batch*1500, 2d]."""
    _need(enc_out, torch.bfloat16, "enc_out")
    batch = enc_out.shape[0]
    d = dims.d_model
    kv = torch.empty((len(layers), batch * N_TOKENS, 2 * d), dtype=torch.bfloat16, device=enc_out.device)
    arr = (_lib.wb_cross_kv_weights * max(1, len(layers)))()
    for i, (w, b) in enumerate(layers):
        arr[i] = _lib.wb_cross_kv_weights(w.data_ptr(), b.data_ptr())
    ds = dims_struct(dims)
    call("wb_cross_kv", _p(enc_out), batch, ctypes.byref(ds), len(layers), arr, _p(kv), _stream(stream))
    return kv


def profile_begin() -> None:
    """Start timing every libwb kernel launch (CUDA events on the launch stream)."""
    call("wb_profile_begin")


def profile_end() -> dict:
    """Stop timing; {kernel class: (summed device ms, kernels launched)}."""
    n = 32
    names = (ctypes.c_char_p * n)()
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    k = load().wb_profile_end(n, names, ms, cnt)
    return {names[i].decode(): (ms[i], cnt[i]) for i in range(min(k, n)) if cnt[i] > 0}


def check_device_error(stream=None) -> int:
    """Synchronize, read and clear the device error words; 0 when no kernel reported a fault.

    A recorded timeout (bit 0) or, in a debug build, a failed bounds check (bit 1) is returned
    as the raw word (site in bits 8..15) rather than raised; a failed synchronization raises
    WbError."""
    word = ctypes.c_uint32(0)
    st = load().wb_check_device_error(_stream(stream), ctypes.byref(word))
    if st not in (WB_OK, WB_ETIMEOUT, _lib.WB_EBOUNDS):
        raise WbError("wb_check_device_error", st)
    return word.value


def selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait diagnostic: a wait that nothing satisfies gives up after ~2 s and
    records a timeout at site WB_SELFTEST_WAIT_SITE (read it back with check_device_error)."""
    call("wb_selftest_wait_timeout", _stream(stream))


# --------------------------------- weights ------------------------------------
@dataclasses.dataclass
class StemWeights:
    conv1_w: torch.Tensor   # bf16 [3, d, n_mels]
    conv1_b: torch.Tensor   # f32 [d]
    conv2_w: torch.Tensor   # bf16 [3, d, d]
    conv2_b: torch.Tensor

    def struct(self) -> _lib.wb_stem_weights:
        self._s = _lib.wb_stem_weights(self.conv1_w.data_ptr(), self.conv1_b.data_ptr(), self.conv2_w.data_ptr(),
                                       self.conv2_b.data_ptr())
        return self._s


@dataclasses.dataclass
class LayerWeights:
    ln1_g: torch.Tensor
    ln1_b: torch.Tensor
    w_qkv: torch.Tensor      # bf16 [3d, d]
    b_qkv: torch.Tensor      # f32 [3d]
    w_out: torch.Tensor
    b_out: torch.Tensor
    ln2_g: torch.Tensor
    ln2_b: torch.Tensor
    w_fc1: torch.Tensor
    b_fc1: torch.Tensor
    w_fc2: torch.Tensor
    b_fc2: torch.Tensor
    fp8: dict = dataclasses.field(default_factory=dict)   # name -> (codes, scale) for E4M3 copies
    ln_fold: dict = dataclasses.field(default_factory=dict)   # "w_qkv" / "w_fc1" -> (w_ln, c, b_ln)


@dataclasses.dataclass
class EncoderWeights:
    layers: list
    ln_post_g: torch.Tensor
    ln_post_b: torch.Tensor

    def quantize(self, names=("w_qkv", "w_fc1", "w_fc2", "w_out")):
        """Make E4M3 copies (per-tensor scale) of the named weights of every layer."""
        for L in self.layers:
            for n in names:
                if n not in L.fp8:
                    L.fp8[n] = quantize_fp8(getattr(L, n))

    def fold_layernorm(self):
        """Fold LN1 into the QKV weights and LN2 into the FC1 weights of every layer (bf16 sites then
        skip their LayerNorm pass)."""
        for L in self.layers:
            if "w_qkv" not in L.ln_fold:
                L.ln_fold["w_qkv"] = fold_layernorm(L.w_qkv, L.b_qkv, L.ln1_g, L.ln1_b)
            if "w_fc1" not in L.ln_fold:
                L.ln_fold["w_fc1"] = fold_layernorm(L.w_fc1, L.b_fc1, L.ln2_g, L.ln2_b)

    def layer_array(self, precision):
        qkv8, out8, ffn8 = precision[0] == WB_E4M3, precision[2] == WB_E4M3, precision[4] == WB_E4M3
        arr = (_lib.wb_layer_weights * max(1, len(self.layers)))()
        for i, L in enumerate(self.layers):
            def pick(name, use8):
                if use8:
                    if name not in L.fp8:
                        raise ValueError(f"layer {i}: no E4M3 copy of {name}; call EncoderWeights.quantize()")
                    q, s = L.fp8[name]
                    return q.data_ptr(), s.data_ptr()
                return getattr(L, name).data_ptr(), None
            wq, sq = pick("w_qkv", qkv8)
            wo, so = pick("w_out", out8)
            w1, s1 = pick("w_fc1", ffn8)
            w2, s2 = pick("w_fc2", ffn8)
            def fold(name):
                f = L.ln_fold.get(name)
                return tuple(t.data_ptr() for t in f) if f is not None else (None, None, None)
            arr[i] = _lib.wb_layer_weights(L.ln1_g.data_ptr(), L.ln1_b.data_ptr(), wq, L.b_qkv.data_ptr(), sq,
                                           wo, L.b_out.data_ptr(), so, L.ln2_g.data_ptr(), L.ln2_b.data_ptr(),
                                           w1, L.b_fc1.data_ptr(), s1, w2, L.b_fc2.data_ptr(), s2,
                                           *fold("w_qkv"), *fold("w_fc1"))
        self._arr = arr
        return arr


def upload_weights(w: dict, device="cuda", fold_ln: bool = True):
    """Host weight dict (HF layout, float32 arrays) -> (StemWeights, EncoderWeights) on the device.
    fold_ln: also make the LayerNorm folds of every layer (EncoderWeights.fold_layernorm)."""
    def f32(a):
        return torch.as_tensor(a, dtype=torch.float32).to(device).contiguous()

    def bf16(a):
        return torch.as_tensor(a, dtype=torch.float32).to(device).to(torch.bfloat16).contiguous()

    stem = StemWeights(pack_conv_weight(f32(w["conv1_w"])), f32(w["conv1_b"]),
                       pack_conv_weight(f32(w["conv2_w"])), f32(w["conv2_b"]))
    layers = []
    for L in w["layers"]:
        d = L["wq"].shape[0]
        zeros = torch.zeros(d, dtype=torch.float32)
        b_qkv = torch.cat([torch.as_tensor(L["bq"]), zeros, torch.as_tensor(L["bv"])])
        w_qkv = torch.cat([torch.as_tensor(L["wq"]), torch.as_tensor(L["wk"]), torch.as_tensor(L["wv"])])
        layers.append(LayerWeights(
            f32(L["ln1_g"]), f32(L["ln1_b"]), bf16(w_qkv), f32(b_qkv), bf16(L["wo"]), f32(L["bo"]),
            f32(L["ln2_g"]), f32(L["ln2_b"]), bf16(L["w1"]), f32(L["b1"]), bf16(L["w2"]), f32(L["b2"])))
    enc = EncoderWeights(layers, f32(w["ln_post_g"]), f32(w["ln_post_b"]))
    if fold_ln:
        enc.fold_layernorm()
    return stem, enc


class Pipeline:
    """audio -> log-mel -> conv stem -> encoder on one stream, with persistent workspaces."""

    def __init__(self, dims, stem: StemWeights, enc: EncoderWeights, batch: int, precision=PRESET_BF16,
                 device="cuda"):
        self.dims, self.stem, self.enc, self.batch, self.precision = dims, stem, enc, batch, precision
        if WB_E4M3 in precision:
            enc.quantize()
        ds = dims_struct(dims)
        self.ws_mel = _workspace(logmel_workspace_bytes(batch, dims.n_mels), device)
        self.ws_stem = _workspace(load().wb_conv_stem_workspace_bytes(ctypes.byref(ds), batch), device)
        self.ws_enc = _workspace(encoder_workspace_bytes(dims, batch, precision), device)
        self.mel = torch.empty((batch, dims.n_mels, N_FRAMES), dtype=torch.float32, device=device)
        self.x0 = torch.empty((batch, N_TOKENS, dims.d_model), dtype=torch.bfloat16, device=device)
        self.out = torch.empty((batch, N_TOKENS, dims.d_model), dtype=torch.bfloat16, device=device)

    def capture(self, audio: torch.Tensor, chunk_stride: int = CHUNK_SAMPLES,
                n_chunks: int | None = None) -> "torch.cuda.CUDAGraph":
        """Record the three library calls on the fixed device buffer ``audio`` into a CUDA graph.

        ``graph.replay()`` then recomputes ``self.out`` from the buffer's current contents with
        one launch instead of ~240 (the calls synchronize nothing and allocate nothing, so
        they can be captured; two eager warm-up calls run first).  The graph reads and writes
        this pipeline's buffers: keep the Pipeline (and ``audio``) alive while it is replayed."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                self(audio, chunk_stride, n_chunks)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self(audio, chunk_stride, n_chunks)
        return graph

    def __call__(self, audio: torch.Tensor, chunk_stride: int = CHUNK_SAMPLES, n_chunks: int | None = None,
                 stream=None, out: torch.Tensor | None = None) -> torch.Tensor:
        n = self.batch if n_chunks is None else n_chunks
        dst = self.out if out is None else out
        logmel(audio, n, self.dims.n_mels, chunk_stride, out=self.mel[:n], workspace=self.ws_mel, stream=stream)
        conv_stem(self.mel[:n], self.dims, self.stem, out=self.x0[:n], workspace=self.ws_stem, stream=stream)
        encoder_forward(self.x0[:n], self.dims, self.enc, self.precision, out=dst[:n], workspace=self.ws_enc,
                        stream=stream)
        return dst[:n]

    def run_host(self, host_in: list, host_out: list, chunk_stride: int = CHUNK_SAMPLES, overlap: bool = True) -> None:
        """Encode a sequence of full batches held in pinned host memory through wb_encode_host.

        host_in[i]: pinned float32 audio of batch i (as for __call__); host_out[i]: pinned bf16
        [batch, 1500, d] that receives batch i's encoder output.  The library copies each batch up,
        runs the three calls and copies the result back; with ``overlap`` the copies run on two
        copy streams against two device input and two device output buffers, so they overlap
        the compute of the neighbouring batches.  Returns with all work queued on the current
        stream (synchronize it to wait for the last download)."""
        n = len(host_in)
        if len(host_out) != n:
            raise ValueError("host_in and host_out differ in length")
        if n == 0:
            return
        for t in host_in:
            if t.dtype != torch.float32 or t.is_cuda or not t.is_contiguous() or t.shape != host_in[0].shape:
                raise ValueError("host_in: contiguous float32 host tensors of one shape expected")
        for t in host_out:
            if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(self.out.shape):
                raise ValueError(f"host_out: contiguous bf16 host tensors of shape {tuple(self.out.shape)} expected")
        if not hasattr(self, "_copy"):
            self._copy = (torch.cuda.Stream(), torch.cuda.Stream())
            self._out2 = torch.empty_like(self.out)
            self._dev_in = None
        if self._dev_in is None or self._dev_in[0].shape != host_in[0].shape:
            self._dev_in = [torch.empty(host_in[0].shape, dtype=torch.float32, device=self.out.device) for _ in range(2)]
        ds, pr = dims_struct(self.dims), precision_struct(self.precision)
        layers = self.enc.layer_array(self.precision)
        ln = _lib.wb_ln_weights(self.enc.ln_post_g.data_ptr(), self.enc.ln_post_b.data_ptr())
        stem = self.stem.struct()
        hp = _lib.wb_host_pipeline()
        hp.dims, hp.batch, hp.samples_per_batch, hp.chunk_stride = ds, self.batch, host_in[0].numel(), chunk_stride
        hp.stem, hp.layers, hp.ln_post, hp.precision = ctypes.pointer(stem), layers, ctypes.pointer(ln), pr
        hp.dev_audio[0], hp.dev_audio[1] = self._dev_in[0].data_ptr(), self._dev_in[1].data_ptr()
        hp.dev_mel, hp.dev_x0 = self.mel.data_ptr(), self.x0.data_ptr()
        hp.dev_out[0], hp.dev_out[1] = self.out.data_ptr(), self._out2.data_ptr()
        hp.ws_mel, hp.ws_mel_bytes = self.ws_mel.data_ptr(), self.ws_mel.numel()
        hp.ws_stem, hp.ws_stem_bytes = self.ws_stem.data_ptr(), self.ws_stem.numel()
        hp.ws_enc, hp.ws_enc_bytes = self.ws_enc.data_ptr(), self.ws_enc.numel()
        if overlap:
            hp.upload_stream, hp.download_stream = self._copy[0].cuda_stream, self._copy[1].cuda_stream
        ins = (ctypes.c_void_p * n)(*[t.data_ptr() for t in host_in])
        outs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in host_out])
        call("wb_encode_host", ctypes.byref(hp), ins, outs, n, _stream())
