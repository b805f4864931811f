"""Log-mel front end in float64 (oracle; test infrastructure only).

Follows the whisper-blaze showcase site, "The Solution" (mel_spectrogram.cu
card: STFT, 128-bin mel filterbank, overlapping-chunk mode for long audio) and
"The Approach" ("Kill the CPU preprocessor"), with the constants the
workload fixes: n_fft 400 with a periodic Hann window, hop 160, reflect-padded
centre framing, Slaney mel bins over 0-8 kHz, the last frame dropped (3000
frames per 30 s chunk), log10(max(x, 1e-10)), clamp to (chunk max - 8), then
(x + 4) / 4.

Readings where the pages are silent (each is listed in the design notes):
  * power spectrum |X|^2 (not magnitude);
  * reflect padding mirrors WITHOUT repeating the edge sample;
  * the dropped frame is the last one, t = 3000;
  * Slaney scale with area normalisation 2 / (f[m+2] - f[m]);
  * the clamp maximum is taken over ONE chunk's C x 3000 values;
  * long audio is cut into 30 s windows at a 25 s stride, zero-filled past
    the end.
"""
from __future__ import annotations

import numpy as np

SAMPLE_RATE = 16000
N_FFT = 400
HOP = 160
N_FRAMES = 3000
CHUNK_SAMPLES = 480000
CHUNK_STRIDE = 400000          # long-form: 25 s stride
N_BINS = N_FFT // 2 + 1        # 201 one-sided bins


def n_chunks_for(n_samples: int, chunk: int = CHUNK_SAMPLES, stride: int = CHUNK_STRIDE) -> int:
    """Number of windows needed so that every sample lies in some window."""
    if n_samples <= chunk:
        return 1
    return 1 + -(-(n_samples - chunk) // stride)


def chunk_audio(samples: np.ndarray, chunk: int = CHUNK_SAMPLES, stride: int = CHUNK_STRIDE,
                n_chunks: int | None = None) -> np.ndarray:
    """Window c covers samples [c*stride, c*stride + chunk), zeros past the end."""
    samples = np.asarray(samples)
    if n_chunks is None:
        n_chunks = n_chunks_for(len(samples), chunk, stride)
    out = np.zeros((n_chunks, chunk), dtype=samples.dtype)
    for c in range(n_chunks):
        seg = samples[c * stride: c * stride + chunk]
        out[c, :len(seg)] = seg
    return out


def reflect_pad(x: np.ndarray, p: int) -> np.ndarray:
    """x[-j] = x[j] and x[N-1+j] = x[N-1-j] for j = 1..p (edge not repeated)."""
    x = np.asarray(x, dtype=np.float64)
    left = x[1:p + 1][::-1]
    right = x[len(x) - 1 - p:len(x) - 1][::-1]
    return np.concatenate([left, x, right])


def hann_periodic(n: int = N_FFT) -> np.ndarray:
    """Periodic Hann window w[i] = 0.5 - 0.5 cos(2 pi i / n), i = 0..n-1."""
    i = np.arange(n, dtype=np.float64)
    return 0.5 - 0.5 * np.cos(2.0 * np.pi * i / n)


def dft_matrices(n_fft: int = N_FFT):
    """Real and imaginary parts of e^{-2 pi i k j / n_fft}, shape [n_fft, n_fft//2+1].

    The phase index (k*j mod n_fft) is reduced exactly in integers first.
    """
    j = np.arange(n_fft)[:, None]
    k = np.arange(n_fft // 2 + 1)[None, :]
    ang = 2.0 * np.pi * ((j * k) % n_fft) / n_fft
    return np.cos(ang), -np.sin(ang)


def frames(x: np.ndarray) -> np.ndarray:
    """Centre framing of one chunk: [n_frames+1, N_FFT] rows of the padded signal."""
    xp = reflect_pad(x, N_FFT // 2)
    n = 1 + (len(xp) - N_FFT) // HOP
    idx = np.arange(n)[:, None] * HOP + np.arange(N_FFT)[None, :]
    return xp[idx]


def stft(x: np.ndarray):
    """Windowed real DFT of every frame (last frame dropped): (re, im) [3000, 201]."""
    fr = frames(x) * hann_periodic()[None, :]
    cos_m, msin_m = dft_matrices()
    re = fr @ cos_m
    im = fr @ msin_m
    return re[:-1], im[:-1]


def power_spectrum(x: np.ndarray) -> np.ndarray:
    """P[t, k] = |X[t, k]|^2, [3000, 201]."""
    re, im = stft(x)
    return re * re + im * im


def hz_to_mel(f):
    """Slaney mel scale: linear 3f/200 below 1 kHz, logarithmic above (27 mels per ln 6.4)."""
    f = np.asarray(f, dtype=np.float64)
    lin = 3.0 * f / 200.0
    logpart = 15.0 + 27.0 * np.log(np.maximum(f, 1e-300) / 1000.0) / np.log(6.4)
    return np.where(f < 1000.0, lin, logpart)


def mel_to_hz(m):
    """Inverse of hz_to_mel."""
    m = np.asarray(m, dtype=np.float64)
    lin = 200.0 * m / 3.0
    logpart = 1000.0 * np.exp((m - 15.0) * np.log(6.4) / 27.0)
    return np.where(m < 15.0, lin, logpart)


def mel_band_edges(n_mels: int, fmax: float = SAMPLE_RATE / 2) -> np.ndarray:
    """n_mels + 2 frequencies (Hz) equally spaced on the mel scale over [0, fmax]."""
    return mel_to_hz(np.linspace(hz_to_mel(0.0), hz_to_mel(fmax), n_mels + 2))


def mel_filterbank(n_mels: int, n_fft: int = N_FFT, sr: int = SAMPLE_RATE,
                   fmax: float = SAMPLE_RATE / 2) -> np.ndarray:
    """Slaney-normalised triangular filters, [n_mels, n_fft//2 + 1].

    Filter m rises from edge m to edge m+1 and falls to edge m+2, scaled by
    2 / (edge[m+2] - edge[m]) so that its area over Hz is 1.
    """
    edges = mel_band_edges(n_mels, fmax)
    fk = np.arange(n_fft // 2 + 1, dtype=np.float64) * sr / n_fft
    fb = np.zeros((n_mels, len(fk)))
    for m in range(n_mels):
        lo, ce, hi = edges[m], edges[m + 1], edges[m + 2]
        rising = (fk - lo) / (ce - lo)
        falling = (hi - fk) / (hi - ce)
        fb[m] = np.maximum(0.0, np.minimum(rising, falling)) * (2.0 / (hi - lo))
    return fb


def mel_power(x: np.ndarray, n_mels: int) -> np.ndarray:
    """M[m, t] = sum_k fb[m, k] P[t, k], [n_mels, 3000]."""
    return mel_filterbank(n_mels) @ power_spectrum(x).T


def log_mel(x: np.ndarray, n_mels: int) -> np.ndarray:
    """Whisper log-mel of one 30 s chunk: float64 [n_mels, 3000]."""
    M = mel_power(np.asarray(x, dtype=np.float64), n_mels)
    L = np.log10(np.maximum(M, 1e-10))
    L = np.maximum(L, L.max() - 8.0)
    return (L + 4.0) / 4.0


def log_mel_batch(chunks: np.ndarray, n_mels: int) -> np.ndarray:
    """log_mel of every row of a [B, 480000] array: [B, n_mels, 3000]."""
    return np.stack([log_mel(c, n_mels) for c in chunks])
