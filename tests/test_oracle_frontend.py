"""Pins of the oracle's log-mel front end against closed forms, invariants and
library special cases (numpy's FFT and padding).  CPU only."""
import numpy as np
import pytest

from oracle import frontend as fe
import synthetic


def test_reflect_pad_matches_numpy_reflect():
    x = np.random.default_rng(1).normal(size=1000)
    np.testing.assert_array_equal(fe.reflect_pad(x, 200), np.pad(x, 200, mode="reflect"))


def test_frame_geometry_centre_and_count():
    x = np.arange(fe.CHUNK_SAMPLES, dtype=np.float64)
    fr = fe.frames(x)
    assert fr.shape == (3001, 400)              # 1 + (480400 - 400) / 160
    # frame t is centred on sample 160 t (away from the reflected edge)
    for t in (2, 17, 1500, 2998):
        assert fr[t, 200] == 160 * t
    re, im = fe.stft(np.zeros(fe.CHUNK_SAMPLES))
    assert re.shape == (3000, 201) and im.shape == (3000, 201)   # last frame dropped


def test_stft_matches_numpy_rfft():
    x = synthetic.tone_chunk(7).astype(np.float64)
    re, im = fe.stft(x)
    fr = fe.frames(x)[:-1] * np.hanning(401)[:-1][None, :]      # periodic Hann == first 400 of a 401 symmetric one
    ref = np.fft.rfft(fr, axis=1)
    scale = np.abs(ref).max()
    assert np.max(np.abs(re - ref.real)) < 1e-12 * scale
    assert np.max(np.abs(im - ref.imag)) < 1e-12 * scale


def test_hann_is_periodic():
    w = fe.hann_periodic(400)
    assert w[0] == 0.0 and abs(w[200] - 1.0) < 1e-15
    assert abs(w.sum() - 200.0) < 1e-9              # sum of a periodic Hann of length N is N/2
    np.testing.assert_allclose(w[1:], w[1:][::-1], atol=1e-15)   # symmetric about n = 200


@pytest.mark.parametrize("amp", [0.1, 0.3])
def test_tone_on_bin_25_closed_form(amp):
    # 1000 Hz = bin 25 (40 Hz bins).  With a periodic Hann the windowed DFT of a
    # pure tone has exactly three nonzero bins: |X[k0]| = 100 A, |X[k0+-1]| = 50 A.
    n = np.arange(fe.CHUNK_SAMPLES)
    x = amp * np.sin(2 * np.pi * 1000.0 * n / fe.SAMPLE_RATE)
    P = fe.power_spectrum(x)[2:2998]           # interior frames only
    np.testing.assert_allclose(P[:, 25], (100 * amp) ** 2, rtol=1e-10)
    np.testing.assert_allclose(P[:, 24], (50 * amp) ** 2, rtol=1e-10)
    np.testing.assert_allclose(P[:, 26], (50 * amp) ** 2, rtol=1e-10)
    others = np.delete(P, [24, 25, 26], axis=1)
    assert others.max() < 1e-20 * (100 * amp) ** 2 * 1e6


def test_dc_closed_form():
    c = 0.25
    re, im = fe.stft(np.full(fe.CHUNK_SAMPLES, c))
    np.testing.assert_allclose(re[:, 0], 200 * c, rtol=1e-12)
    np.testing.assert_allclose(re[:, 1], -100 * c, rtol=1e-12)
    assert np.abs(im[:, :2]).max() < 1e-12
    assert np.abs(re[:, 2:]).max() < 1e-11 and np.abs(im[:, 2:]).max() < 1e-11


def test_parseval():
    x = synthetic.tone_chunk(3).astype(np.float64)
    re, im = fe.stft(x)
    P = re ** 2 + im ** 2
    lhs = P[:, 0] + 2 * P[:, 1:200].sum(1) + P[:, 200]
    wx = fe.frames(x)[:-1] * fe.hann_periodic()[None, :]
    rhs = 400.0 * (wx ** 2).sum(1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-11)


def test_slaney_scale_points():
    assert fe.hz_to_mel(1000.0) == pytest.approx(15.0, abs=1e-12)
    assert fe.hz_to_mel(500.0) == pytest.approx(7.5, abs=1e-12)
    assert fe.hz_to_mel(6400.0) == pytest.approx(42.0, abs=1e-12)      # 27 mels per factor 6.4
    assert fe.hz_to_mel(8000.0) == pytest.approx(45.2456, abs=1e-4)
    f = np.array([0.0, 37.0, 999.0, 1000.0, 1234.5, 7999.0])
    np.testing.assert_allclose(fe.mel_to_hz(fe.hz_to_mel(f)), f, atol=1e-9)
    edges = fe.mel_band_edges(128)
    assert edges[0] == 0.0 and edges[-1] == pytest.approx(8000.0, abs=1e-9)


@pytest.mark.parametrize("n_mels", [80, 128])
def test_mel_triangles_partition_of_unity_and_unit_area(n_mels):
    # Fine frequency grid (0.1 Hz): un-normalised triangles sharing vertices sum
    # to exactly 1 between the first and last centre; each normalised filter
    # has unit area over Hz.
    n_fft = 160000
    fb = fe.mel_filterbank(n_mels, n_fft=n_fft)
    df = fe.SAMPLE_RATE / n_fft
    edges = fe.mel_band_edges(n_mels)
    tri = fb * ((edges[2:] - edges[:-2]) / 2.0)[:, None]
    fk = np.arange(fb.shape[1]) * df
    inside = (fk >= edges[1]) & (fk <= edges[-2])
    np.testing.assert_allclose(tri[:, inside].sum(0), 1.0, atol=1e-9)
    area = fb.sum(1) * df
    np.testing.assert_allclose(area, 1.0, atol=2e-3)
    assert tri.max() <= 1.0 + 1e-12


@pytest.mark.parametrize("n_mels,last_row_sum,first_wide,wmin,wmax",
                         [(80, 0.9970, 41, 74.5, 591.0), (128, 0.9974, 84, 46.8, 377.0)])
def test_mel_filterbank_at_40hz_bins(n_mels, last_row_sum, first_wide, wmin, wmax):
    fb = fe.mel_filterbank(n_mels)
    assert fb.shape == (n_mels, 201)
    assert (fb.max(1) > 0).all()                         # no empty rows
    sums = fb.sum(1) * 40.0
    assert sums[-1] == pytest.approx(last_row_sum, abs=1e-3)
    assert np.all(np.abs(sums[first_wide:] - 1.0) < 0.05)
    edges = fe.mel_band_edges(n_mels)
    widths = edges[2:] - edges[:-2]
    assert widths.min() == pytest.approx(wmin, abs=0.1)
    assert widths.max() == pytest.approx(wmax, abs=1.0)


def test_log_mel_of_silence_is_minus_1p5():
    y = fe.log_mel(synthetic.silence(), 80)
    assert y.shape == (80, 3000)
    assert np.all(y == -1.5)                            # (log10(1e-10) + 4) / 4


def test_half_silence_activates_per_chunk_clamp():
    x = synthetic.half_silence(11)
    y = fe.log_mel(x, 128)
    M = fe.mel_power(x.astype(np.float64), 128)
    top = np.log10(M.max())
    silent = y[:, 1502:]                                 # frames wholly inside the zero half
    np.testing.assert_allclose(silent, (top - 8.0 + 4.0) / 4.0, atol=1e-12)
    assert y.max() == pytest.approx((top + 4.0) / 4.0, abs=1e-12)


def test_clamp_is_per_chunk():
    a = synthetic.tone_chunk(5)
    quiet = (0.001 * synthetic.tone_chunk(6)).astype(np.float32)
    ya = fe.log_mel_batch(np.stack([a, quiet]), 80)
    np.testing.assert_array_equal(ya[1], fe.log_mel(quiet, 80))


def test_long_form_chunking():
    n = 43_200_000
    assert fe.n_chunks_for(n) == 108
    assert fe.n_chunks_for(480000) == 1 and fe.n_chunks_for(480001) == 2
    x = np.arange(1_300_000, dtype=np.float32)
    c = fe.chunk_audio(x)
    assert c.shape == (fe.n_chunks_for(1_300_000), 480000)
    assert c[1, 0] == 400000 and c[2, 0] == 800000
    assert c.shape[0] == 4 and c[3, 0] == 1_200_000
    assert c[3, 99_999] == 1_299_999
    assert np.all(c[3, 100_000:] == 0)                   # zero fill past the end
    assert 107 * 400000 / 16000 == 2675.0                # last long-form window start (s)
