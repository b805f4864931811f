"""The bounds-checked debug build of libwb and canary bytes around every output.

A debug build (-DWB_DEBUG, built here as _build_debug/libwb_debug.so) checks
the index of every kernel load and store that does not go through a TMA tensor
map against the extent of the buffer it addresses, and records a violation in
the device error word instead of touching memory.  These tests run the C-ABI
calls at ragged shapes (sequence lengths 1, 129 and 1500, N = 1152, row counts
that are not multiples of the tile sizes, a zero-filled last long-form window)
on both builds, with every output and workspace placed between guard bytes of a
known pattern, and check that:
  * the debug build reports no bounds error,
  * no guard byte changed in either build (this also covers the TMA stores,
    which the debug checks cannot see),
  * both builds give bitwise the same outputs (the checks change no arithmetic)."""
import ctypes

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu
GUARD = 0xA5
HEAD, TAIL = 256, 4096


class Guarded:
    """A device tensor of the given shape / dtype with guard bytes before and after it."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((HEAD + n + TAIL,), GUARD, dtype=torch.uint8, device="cuda")
        self.t = self.raw[HEAD:HEAD + n].view(dtype).view(*shape) if n else self.raw[HEAD:HEAD].view(dtype)
        self.n = n

    @property
    def p(self):
        return ctypes.c_void_p(self.raw.data_ptr() + HEAD)

    def guards_intact(self) -> bool:
        return bool((self.raw[:HEAD] == GUARD).all()) and bool((self.raw[HEAD + self.n:] == GUARD).all())


@pytest.fixture(scope="module")
def libs(wb):
    from whisper_encoder_gb300 import _lib, build
    rel = _lib.load()
    dbg = _lib.open_library(build.build(debug=True))
    assert rel.wb_debug_build() == 0 and dbg.wb_debug_build() == 1
    return {"release": rel, "debug": dbg}


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check_word(lib):
    word = ctypes.c_uint32(0)
    st = lib.wb_check_device_error(_stream(), ctypes.byref(word))
    return st, word.value


def _run_both(libs, fn):
    """fn(lib) -> list of Guarded outputs; run on both builds, check guards, words and equality."""
    outs = {}
    for name, lib in libs.items():
        g = fn(lib)
        torch.cuda.synchronize()
        st, word = _check_word(lib)
        assert st == 0 and word == 0, (name, st, hex(word))
        for i, b in enumerate(g):
            assert b.guards_intact(), (name, i)
        outs[name] = [b.t.clone() for b in g]
    for a, b in zip(outs["release"], outs["debug"]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    return outs["release"]


def test_logmel_long_form_ragged(libs, wb):
    x = torch.from_numpy(synthetic.long_audio(synthetic.SEED_LONGFORM, 1_300_000)).cuda()
    n, stride = 4, 400000                       # the last window runs past the end (zero fill)
    def fn(lib):
        out = Guarded((n, 80, 3000), torch.float32)
        ws = Guarded((lib.wb_logmel_workspace_bytes(n, 80),), torch.uint8)
        assert lib.wb_logmel(ctypes.c_void_p(x.data_ptr()), x.numel(), stride, n, 80, out.p, ws.p, ws.n,
                             _stream()) == 0
        return [out, ws]
    _run_both(libs, fn)


@pytest.mark.parametrize("T,H", [(1, 2), (129, 1), (1500, 2)])
def test_attention_ragged(libs, T, H):
    g = torch.Generator(device="cuda").manual_seed(T)
    q, k, v = (torch.randn(1, T, 64 * H, device="cuda", generator=g).to(torch.bfloat16) for _ in range(3))
    def fn(lib):
        out = Guarded((1, T, 64 * H), torch.bfloat16)
        ws = Guarded((lib.wb_attention_workspace_bytes(1, T, H),), torch.uint8)
        args = [ctypes.c_void_p(t.data_ptr()) for t in (q, k, v)]
        assert lib.wb_attention(*args, 1, T, H, out.p, ws.p, ws.n, _stream()) == 0
        return [out, ws]
    _run_both(libs, fn)


@pytest.mark.parametrize("M,N,K,gelu,resid", [(129, 1152, 384, 0, False), (129, 1152, 384, 1, False),
                                              (1500, 1152, 640, 0, True), (33, 256, 64, 1, True)])
def test_linear_bf16_ragged(libs, M, N, K, gelu, resid):
    g = torch.Generator(device="cuda").manual_seed(M + N)
    a = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    bias = torch.randn(N, device="cuda", generator=g)
    r = torch.randn(M, N, device="cuda", generator=g).to(torch.bfloat16) if resid else None
    def fn(lib):
        out = Guarded((M, N), torch.bfloat16)
        assert lib.wb_linear(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(w.data_ptr()), M, N, K, 0,
                             ctypes.c_void_p(bias.data_ptr()), None, None, gelu,
                             ctypes.c_void_p(r.data_ptr()) if r is not None else None, out.p, _stream()) == 0
        return [out]
    _run_both(libs, fn)


def test_linear_e4m3_ragged(libs, wb):
    M, N, K = 257, 1152, 640
    g = torch.Generator(device="cuda").manual_seed(9)
    qa, sa = wb.quantize_fp8(torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16))
    qw, sw = wb.quantize_fp8((torch.randn(N, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16))
    def fn(lib):
        out = Guarded((M, N), torch.bfloat16)
        assert lib.wb_linear(ctypes.c_void_p(qa.data_ptr()), ctypes.c_void_p(qw.data_ptr()), M, N, K, 1, None,
                             ctypes.c_void_p(sa.data_ptr()), ctypes.c_void_p(sw.data_ptr()), 1, None, out.p,
                             _stream()) == 0
        return [out]
    _run_both(libs, fn)


@pytest.mark.parametrize("rows,d", [(129, 384), (1, 1280), (3001, 640)])
def test_norms_and_codecs_ragged(libs, rows, d):
    g = torch.Generator(device="cuda").manual_seed(rows)
    x = torch.randn(rows, d, device="cuda", generator=g).to(torch.bfloat16)
    res = torch.randn(rows, d, device="cuda", generator=g).to(torch.bfloat16)
    gam = 1 + 0.1 * torch.randn(d, device="cuda", generator=g)
    bet = 0.1 * torch.randn(d, device="cuda", generator=g)
    rpi = max(1, rows // 3)
    items = (rows + rpi - 1) // rpi
    n = rows * d - 7                             # a ragged element count for the codecs
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    def fn(lib):
        y, tot = Guarded((rows, d), torch.bfloat16), Guarded((rows, d), torch.bfloat16)
        assert lib.wb_layernorm(P(x), P(res), P(gam), P(bet), rows, d, 1e-5, y.p, tot.p, _stream()) == 0
        yr, totr = Guarded((rows, d), torch.bfloat16), Guarded((rows, d), torch.bfloat16)
        assert lib.wb_rmsnorm(P(x), P(res), P(gam), rows, d, 1e-5, yr.p, totr.p, _stream()) == 0
        q, am, st = Guarded((rows, d), torch.uint8), Guarded((items,), torch.float32), Guarded((rows, 2), torch.float32)
        assert lib.wb_layernorm_e4m3(P(x), P(gam), P(bet), rows, d, 1e-5, rpi, q.p, am.p, st.p, _stream()) == 0
        q8, s8 = Guarded((n,), torch.uint8), Guarded((1,), torch.float32)
        assert lib.wb_quantize_fp8(P(x), n, q8.p, s8.p, _stream()) == 0
        d8 = Guarded((n,), torch.bfloat16)
        assert lib.wb_dequantize_fp8(q8.p, s8.p, n, d8.p, _stream()) == 0
        q5, s5 = Guarded((n,), torch.uint8), Guarded((1,), torch.float32)
        assert lib.wb_quantize_e5m2(P(x), n, q5.p, s5.p, _stream()) == 0
        return [y, tot, yr, totr, q, am, st, q8, s8, d8, q5, s5]
    _run_both(libs, fn)


@pytest.mark.parametrize("precision_name", ["PRESET_BF16", "PRESET_MIXED_FP8"])
def test_stem_and_encoder_tiny(libs, wb, precision_name):
    dims = synthetic.TINY
    stem, enc = wb.upload_weights(synthetic.encoder_weights(dims, synthetic.SEED_TINY, "f32"))
    precision = getattr(wb, precision_name)
    if precision != wb.PRESET_BF16:
        enc.quantize()
    B = 3
    mel = torch.from_numpy(np.random.default_rng(3).uniform(-1.5, 1.5, (B, dims.n_mels, 3000)).astype(np.float32)).cuda()
    ds, pr = wb.api.dims_struct(dims), wb.api.precision_struct(precision)
    layers = enc.layer_array(precision)
    ln = wb._lib.wb_ln_weights(enc.ln_post_g.data_ptr(), enc.ln_post_b.data_ptr())
    st = stem.struct()
    def fn(lib):
        x0 = Guarded((B, 1500, dims.d_model), torch.bfloat16)
        wss = Guarded((lib.wb_conv_stem_workspace_bytes(ctypes.byref(ds), B),), torch.uint8)
        assert lib.wb_conv_stem(ctypes.c_void_p(mel.data_ptr()), B, ctypes.byref(ds), ctypes.byref(st), x0.p, wss.p,
                                wss.n, _stream()) == 0
        out = Guarded((B, 1500, dims.d_model), torch.bfloat16)
        wse = Guarded((lib.wb_encoder_workspace_bytes(ctypes.byref(ds), B, ctypes.byref(pr)),), torch.uint8)
        assert lib.wb_encoder_forward(x0.p, B, ctypes.byref(ds), layers, ctypes.byref(ln), ctypes.byref(pr), 0,
                                      dims.n_layers, 1, out.p, wse.p, wse.n, _stream()) == 0
        return [x0, wss, out, wse]
    _run_both(libs, fn)


def test_cross_kv_tiny(libs, wb):
    dims = synthetic.TINY
    d = dims.d_model
    g = torch.Generator(device="cuda").manual_seed(5)
    enc_out = torch.randn(2, 1500, d, device="cuda", generator=g).to(torch.bfloat16)
    ws = [((torch.randn(2 * d, d, device="cuda", generator=g) * 0.05).to(torch.bfloat16),
           torch.randn(2 * d, device="cuda", generator=g)) for _ in range(2)]
    arr = (wb._lib.wb_cross_kv_weights * 2)(*[wb._lib.wb_cross_kv_weights(w.data_ptr(), b.data_ptr()) for w, b in ws])
    ds = wb.api.dims_struct(dims)
    def fn(lib):
        kv = Guarded((2, 2 * 1500, 2 * d), torch.bfloat16)
        assert lib.wb_cross_kv(ctypes.c_void_p(enc_out.data_ptr()), 2, ctypes.byref(ds), 2, arr, kv.p, _stream()) == 0
        return [kv]
    _run_both(libs, fn)


def test_bounds_check_selftest_reports_in_debug_build_only(libs):
    # the reporting path of a failed check, end to end, without any out-of-range access: the debug
    # build records the bounds bit and the self-test site, the release build records nothing
    from whisper_encoder_gb300 import _lib
    for name, lib in libs.items():
        assert lib.wb_selftest_bounds_check(_stream()) == 0
        st, word = _check_word(lib)
        if name == "debug":
            assert st == _lib.WB_EBOUNDS and word == (2 | (_lib.WB_SELFTEST_BOUNDS_SITE << 8)), (st, hex(word))
            assert _check_word(lib) == (0, 0)            # reading cleared it
        else:
            assert (st, word) == (0, 0)
