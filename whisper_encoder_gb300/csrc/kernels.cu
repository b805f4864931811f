// Bandwidth-bound SIMT kernels of libwb: audio framing prep, constant tables
// (DFT basis, mel filterbank), log-mel clamp/scale, conv-stem re-layout,
// fused residual + LayerNorm, FP8 absmax / quantise / dequantise.
#include <cuda_fp16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace wb {

// Error word of the bounds checks that debug builds compile into this file's kernels (read and
// cleared by wb_check_device_error through simt_err_ptr()).
__device__ uint32_t g_simt_err;

namespace {

#define WB_IN(idx, len, extent, site) in_bounds(&g_simt_err, (idx), (len), (extent), (site))

constexpr int EW_THREADS = 256;

int grid_for(long long work, int per_block, int cap = 152 * 32) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return static_cast<int>(g);
}

// ---------------------------------------------------------------------------
// Reflect-pad each 30 s chunk by 200 samples (mirror without the edge sample)
// and split every float32 sample exactly into three bf16 parts (hi + mid +
// lo), the operand of the split-precision DFT.  xs: [n_chunks][3][PADDED].
// ---------------------------------------------------------------------------
__global__ void pad_split_kernel(const float* __restrict__ audio, long long n_samples, long long stride,
                                 int n_chunks, __nv_bfloat16* __restrict__ xs) {
  const long long total = static_cast<long long>(n_chunks) * PADDED;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i / PADDED);
    const int j = static_cast<int>(i % PADDED);
    int src = j - PAD;
    if (src < 0) src = -src;
    else if (src >= CHUNK) src = 2 * (CHUNK - 1) - src;
    const long long g = static_cast<long long>(c) * stride + src;
    const float x = g < n_samples ? __ldg(audio + g) : 0.0f;
    const __nv_bfloat16 a = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(a);
    const __nv_bfloat16 b = __float2bfloat16_rn(r1);
    const __nv_bfloat16 e = __float2bfloat16_rn(r1 - __bfloat162float(b));
    const long long o = static_cast<long long>(c) * 3 * PADDED + j;
    if (!WB_IN(o, 2 * PADDED + 1, static_cast<long long>(n_chunks) * 3 * PADDED, SITE_PAD_SPLIT)) continue;
    xs[o] = a;
    xs[o + PADDED] = b;
    xs[o + 2 * PADDED] = e;
  }
}

// Windowed real-DFT basis, [3 parts][512 rows][400]: rows 256*t + c hold, for
// tile t, c < 128: w[k] cos(2 pi bin k / 400) and c >= 128: -w[k] sin(...),
// bin = 128 t + (c mod 128); bins above 200 are zero.  The phase index
// bin*k mod 400 is reduced exactly in integers; values are formed in float (the
// three bf16 parts that follow carry 24 bits, a float's precision) and split.
__global__ void dft_basis_kernel(__nv_bfloat16* __restrict__ basis) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= DFT_ROWS * N_FFT) return;
  const int row = idx / N_FFT, k = idx % N_FFT;
  const int tile = row / 256, col = row % 256;
  const int bin = tile * 128 + (col & 127);
  float v = 0.0f;
  if (bin <= N_FFT / 2) {
    const float w = 0.5f - 0.5f * cospif(static_cast<float>(k) / 200.0f);
    const int ph = (bin * k) % N_FFT;
    float s, c;
    sincospif(static_cast<float>(ph) / 200.0f, &s, &c);
    v = w * (col >= 128 ? -s : c);
  }
  const __nv_bfloat16 a = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(a);
  const __nv_bfloat16 b = __float2bfloat16_rn(r1);
  const __nv_bfloat16 e = __float2bfloat16_rn(r1 - __bfloat162float(b));
  if (!WB_IN((2 * DFT_ROWS + row) * N_FFT + k, 1, 3 * DFT_ROWS * N_FFT, SITE_DFT_BASIS)) return;
  basis[(0 * DFT_ROWS + row) * N_FFT + k] = a;
  basis[(1 * DFT_ROWS + row) * N_FFT + k] = b;
  basis[(2 * DFT_ROWS + row) * N_FFT + k] = e;
}

__device__ float hz_to_mel(float f) {
  return f < 1000.0f ? 3.0f * f / 200.0f : 15.0f + 27.0f * logf(f / 1000.0f) / logf(6.4f);
}
__device__ float mel_to_hz(float m) {
  return m < 15.0f ? 200.0f * m / 3.0f : 1000.0f * expf((m - 15.0f) * logf(6.4f) / 27.0f);
}

// Slaney mel filterbank over 0-8 kHz at the 201 bins of a 400-point DFT,
// [2 parts][128 rows][256 bins] (rows >= n_mels and bins > 200 are zero):
// triangle from edge m to edge m+2 peaking at edge m+1, area-normalised by
// 2 / (edge[m+2] - edge[m]); edges equally spaced on the Slaney mel scale.
__global__ void mel_fb_kernel(__nv_bfloat16* __restrict__ fbs, int n_mels) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= MEL_ROWS * N_BIN_PAD) return;
  const int m = idx / N_BIN_PAD, k = idx % N_BIN_PAD;
  float v = 0.0f;
  if (m < n_mels && k <= N_FFT / 2) {
    const float step = hz_to_mel(8000.0f) / static_cast<float>(n_mels + 1);
    const float lo = mel_to_hz(m * step), ce = mel_to_hz((m + 1) * step), hi = mel_to_hz((m + 2) * step);
    const float f = 40.0f * k;
    const float up = (f - lo) / (ce - lo), dn = (hi - f) / (hi - ce);
    v = fmaxf(0.0f, fminf(up, dn)) * 2.0f / (hi - lo);
  }
  const __nv_bfloat16 a = __float2bfloat16_rn(v);
  const __nv_bfloat16 b = __float2bfloat16_rn(v - __bfloat162float(a));
  if (!WB_IN((MEL_ROWS + m) * N_BIN_PAD + k, 1, 2 * MEL_ROWS * N_BIN_PAD, SITE_MEL_FB)) return;
  fbs[m * N_BIN_PAD + k] = a;
  fbs[(MEL_ROWS + m) * N_BIN_PAD + k] = b;
}

// y = (max(L, log10(max(chunk max, 1e-10)) - 8) + 4) / 4, in place on [n_chunks][n_mels*3000].
__global__ void logmel_post_kernel(float* __restrict__ out, const float* __restrict__ mel_max, int per_chunk) {
  const int b = blockIdx.y;
  const float thr = log10f(fmaxf(mel_max[b], 1e-10f)) - 8.0f;
  float4* p = reinterpret_cast<float4*>(out + static_cast<long long>(b) * per_chunk);
  const int n4 = per_chunk / 4;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += gridDim.x * blockDim.x) {
    if (!WB_IN(static_cast<long long>(b) * per_chunk + 4LL * i, 4, static_cast<long long>(gridDim.y) * per_chunk,
               SITE_LOGMEL_POST))
      continue;
    float4 v = p[i];
    v.x = (fmaxf(v.x, thr) + 4.0f) * 0.25f;
    v.y = (fmaxf(v.y, thr) + 4.0f) * 0.25f;
    v.z = (fmaxf(v.z, thr) + 4.0f) * 0.25f;
    v.w = (fmaxf(v.w, thr) + 4.0f) * 0.25f;
    p[i] = v;
  }
}

// log-mel [B][C][3000] float32 -> time-major bf16 rows 1..3000 of yTp [B][3002][C].
__global__ void stem_transpose_kernel(const float* __restrict__ in, int C, __nv_bfloat16* __restrict__ out) {
  __shared__ float tile[32][33];
  const int b = blockIdx.z, t0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  for (int ty = threadIdx.y; ty < 32; ty += blockDim.y) {
    const int c = c0 + ty, t = t0 + threadIdx.x;
    const long long ii = (static_cast<long long>(b) * C + c) * N_FRAMES + t;
    tile[ty][threadIdx.x] = (c < C && t < N_FRAMES && WB_IN(ii, 1, static_cast<long long>(gridDim.z) * C * N_FRAMES,
                                                           SITE_STEM_T_IN))
                                ? in[ii]
                                : 0.0f;
  }
  __syncthreads();
  for (int ty = threadIdx.y; ty < 32; ty += blockDim.y) {
    const int t = t0 + ty, c = c0 + threadIdx.x;
    const long long oi = (static_cast<long long>(b) * (N_FRAMES + 2) + 1 + t) * C + c;
    if (t < N_FRAMES && c < C && WB_IN(oi, 1, static_cast<long long>(gridDim.z) * (N_FRAMES + 2) * C, SITE_STEM_T_OUT))
      out[oi] = __float2bfloat16_rn(tile[threadIdx.x][ty]);
  }
}

__global__ void zero_rows_kernel(__nv_bfloat16* base, long long row_elems, long long batch_stride, int batch,
                                 int row) {
  const int b = blockIdx.y;
  if (b >= batch) return;
  __nv_bfloat16* p = base + b * batch_stride + row * row_elems;
  for (long long i = blockIdx.x * blockDim.x + threadIdx.x; i < row_elems; i += gridDim.x * blockDim.x)
    if (WB_IN(b * batch_stride + row * row_elems + i, 1, batch * batch_stride, SITE_ZERO_ROWS))
      p[i] = __float2bfloat16_rn(0.0f);
}

// PyTorch Conv1d weight [c_out][c_in][3] float32 -> tap-major bf16 [3][c_out][c_in].
__global__ void pack_conv_kernel(const float* __restrict__ w, int c_out, int c_in, __nv_bfloat16* __restrict__ out) {
  const long long n = static_cast<long long>(c_out) * c_in * 3;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(i % 3);
    const long long oi = i / 3;   // o * c_in + ci
    if (WB_IN(j * static_cast<long long>(c_out) * c_in + oi, 1, n, SITE_PACK_CONV))
      out[j * static_cast<long long>(c_out) * c_in + oi] = __float2bfloat16_rn(w[i]);
  }
}

// ---------------------------------------------------------------------------
// Fused residual + LayerNorm: one warp per row of width NV*VEC*32, the row
// held in registers (exact two-pass mean / variance), 8- or 16-byte loads.
// ---------------------------------------------------------------------------
template <int VEC>
struct VecIO;
template <>
struct VecIO<8> {
  using T = uint4;
};
template <>
struct VecIO<4> {
  using T = uint2;
};

constexpr int LN_WARPS = 8;

template <int NV, int VEC, bool RES>
__device__ __forceinline__ void ln_load(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ res,
                                        long long row, long long rows, int lane, typename VecIO<VEC>::T (&u)[NV],
                                        typename VecIO<VEC>::T (&ur)[NV]) {
  using V = typename VecIO<VEC>::T;
  constexpr int D = NV * VEC * 32;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    if (!WB_IN(row * D + (i * 32 + lane) * VEC, VEC, rows * D, SITE_LN_X)) continue;
    u[i] = __ldg(reinterpret_cast<const V*>(x + row * D + (i * 32 + lane) * VEC));
    if (RES) ur[i] = __ldg(reinterpret_cast<const V*>(res + row * D + (i * 32 + lane) * VEC));
  }
}

// Persistent: warp w normalises the contiguous rows [w*R, (w+1)*R), loading row i+1 before it
// reduces row i so that two rows of loads are in flight per warp.
template <int NV, int VEC, bool RES, bool RMS>
__global__ void __launch_bounds__(LN_WARPS * 32)
    layernorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ res,
                     const float* __restrict__ g, const float* __restrict__ bta, int rows, float eps,
                     __nv_bfloat16* __restrict__ y, __nv_bfloat16* __restrict__ total) {
  constexpr int D = NV * VEC * 32;
  using V = typename VecIO<VEC>::T;
  const int lane = threadIdx.x & 31;
  const long long warp_g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long per = (rows + n_warps - 1) / n_warps;
  const long long r0 = warp_g * per;
  const long long r1 = r0 + per < rows ? r0 + per : rows;
  V u[NV], ur[NV], nu[NV], nur[NV];
  if (r0 < r1) ln_load<NV, VEC, RES>(x, res, r0, rows, lane, u, ur);
  for (long long row = r0; row < r1; ++row) {
    if (row + 1 < r1) ln_load<NV, VEC, RES>(x, res, row + 1, rows, lane, nu, nur);
    float v[NV * VEC];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u[i]);
#pragma unroll
      for (int j = 0; j < VEC; ++j) v[i * VEC + j] = __bfloat162float(h[j]);
      if (RES) {
        const __nv_bfloat16* hr = reinterpret_cast<const __nv_bfloat16*>(&ur[i]);
#pragma unroll
        for (int j = 0; j < VEC; ++j) v[i * VEC + j] += __bfloat162float(hr[j]);
        if (total) {
          V o;
          uint32_t* o32 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
          for (int j = 0; j < VEC / 2; ++j) o32[j] = pack_bf16(v[i * VEC + 2 * j], v[i * VEC + 2 * j + 1]);
          if (WB_IN(row * D + (i * 32 + lane) * VEC, VEC, static_cast<long long>(rows) * D, SITE_LN_Y))
            *reinterpret_cast<V*>(total + row * D + (i * 32 + lane) * VEC) = o;
        }
      }
    }
    float mean = 0.0f;
    if (!RMS) {   // RMSNorm skips the mean (and the beta shift)
      float sm = 0.0f;
#pragma unroll
      for (int i = 0; i < NV * VEC; ++i) sm += v[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      mean = sm * (1.0f / D);
    }
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < NV * VEC; ++i) {
      const float t = v[i] - mean;
      q += t * t;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = rsqrtf(q * (1.0f / D) + eps);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int off = (i * 32 + lane) * VEC;
      if (!WB_IN(off, VEC, D, SITE_LN_GB)) continue;
      // gamma / beta for this lane's VEC columns as 16-byte vector loads (L1-resident, coalesced)
      float gg[VEC], bb[VEC];
#pragma unroll
      for (int j4 = 0; j4 < VEC / 4; ++j4) {
        const float4 g4 = __ldg(reinterpret_cast<const float4*>(g + off) + j4);
        const float4 b4 = RMS ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldg(reinterpret_cast<const float4*>(bta + off) + j4);
        gg[4 * j4 + 0] = g4.x; gg[4 * j4 + 1] = g4.y; gg[4 * j4 + 2] = g4.z; gg[4 * j4 + 3] = g4.w;
        bb[4 * j4 + 0] = b4.x; bb[4 * j4 + 1] = b4.y; bb[4 * j4 + 2] = b4.z; bb[4 * j4 + 3] = b4.w;
      }
      V o;
      uint32_t* o32 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int j = 0; j < VEC / 2; ++j) {
        const float y0 = fmaf((v[i * VEC + 2 * j] - mean) * rstd, gg[2 * j], bb[2 * j]);
        const float y1 = fmaf((v[i * VEC + 2 * j + 1] - mean) * rstd, gg[2 * j + 1], bb[2 * j + 1]);
        o32[j] = pack_bf16(y0, y1);
      }
      if (WB_IN(row * D + off, VEC, static_cast<long long>(rows) * D, SITE_LN_Y))
        *reinterpret_cast<V*>(y + row * D + off) = o;
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      u[i] = nu[i];
      if (RES) ur[i] = nur[i];
    }
  }
}

// ---------------------------------------------------------------------------
// LayerNorm straight to E4M3 codes, in two passes over x (no bf16 output round trip).  The
// per-item scale needs the absmax of the whole item's LayerNorm output before any code can be
// written, so pass 1 computes the row statistics and that absmax (of the bf16-rounded output,
// as the bf16 LayerNorm followed by the quantiser sees it) and pass 2 recomputes the output
// from the statistics and writes code = E4M3_rn_satfinite(bf16(y) * 448 / amax[item]).
// ---------------------------------------------------------------------------
// Packed helpers for the E4M3 LayerNorm: y = fmaf((x - mean) * rstd, g, b) on pairs (lane-wise the
// same IEEE operations as layernorm_kernel's output), then rounded to a bf16 pair.
__device__ __forceinline__ uint64_t ln_affine_x2(uint64_t x2, uint64_t nmean2, uint64_t rstd2, uint64_t g2,
                                                 uint64_t b2) {
  const uint64_t one2 = f32x2_pack(1.0f, 1.0f);
  return f32x2_fma(f32x2_mul(f32x2_fma(x2, one2, nmean2), rstd2), g2, b2);
}
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(uint64_t v) {
  float lo, hi;
  f32x2_unpack(v, lo, hi);
  return pack_bf16(lo, hi);
}
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  return f32x2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Pass 1: stats[row] = (mean, rstd) (two passes over the row held in registers, biased variance,
// as layernorm_kernel), and amax[item] = max |bf16(LN(x; g, b))| over the rows of each item
// (item = row / rows_per_item).  A warp per row, lane t owning columns 128k + 4t .. 4t+3, so that
// the gamma / beta reads of a warp are contiguous; persistent, with the next row loaded while this
// one is reduced.
template <int NK, bool AMAX>
__global__ void __launch_bounds__(LN_WARPS * 32)
    ln_stats_amax_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ g,
                         const float* __restrict__ bta, int rows, float eps, float2* __restrict__ stats,
                         float* __restrict__ amax, int rows_per_item) {
  constexpr int D = NK * 128;
  grid_dependency_wait();
  grid_dependents_launch();
  const int lane = threadIdx.x & 31;
  const long long warp_g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long per = (rows + n_warps - 1) / n_warps;
  const long long r0 = warp_g * per;
  const long long r1 = r0 + per < rows ? r0 + per : rows;
  auto load = [&](long long row, uint2 (&u)[NK]) {
#pragma unroll
    for (int k = 0; k < NK; ++k)
      if (WB_IN(row * D + 128 * k + 4 * lane, 4, static_cast<long long>(rows) * D, SITE_STATS_X))
        u[k] = __ldg(reinterpret_cast<const uint2*>(x + row * D + 128 * k) + lane);
  };
  const int n_items = (rows + rows_per_item - 1) / rows_per_item;
  uint2 u[NK], nu[NK];
  if (r0 < r1) load(r0, u);
  uint32_t run_max2 = 0u;                          // packed bf16 |y| maxima of the current item
  int run_item = r0 < r1 ? static_cast<int>(r0 / rows_per_item) : 0;
  auto flush = [&]() {
    float m = fmaxf(__uint_as_float(run_max2 << 16), __uint_as_float(run_max2 & 0xffff0000u));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0 && m > 0.0f && WB_IN(run_item, 1, n_items, SITE_STATS_AMAX)) atomic_max_nonneg(amax + run_item, m);
  };
  for (long long row = r0; row < r1; ++row) {
    if (row + 1 < r1) load(row + 1, nu);
    float sm = 0.0f;
#pragma unroll
    for (int k = 0; k < NK; ++k)
      sm += (__uint_as_float(u[k].x << 16) + __uint_as_float(u[k].x & 0xffff0000u)) +
            (__uint_as_float(u[k].y << 16) + __uint_as_float(u[k].y & 0xffff0000u));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    const float mean = sm * (1.0f / D);
    float q = 0.0f;
#pragma unroll
    for (int k = 0; k < NK; ++k) {
      const float v[4] = {__uint_as_float(u[k].x << 16), __uint_as_float(u[k].x & 0xffff0000u),
                          __uint_as_float(u[k].y << 16), __uint_as_float(u[k].y & 0xffff0000u)};
#pragma unroll
      for (int j = 0; j < 4; ++j) q = fmaf(v[j] - mean, v[j] - mean, q);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = rsqrtf(q * (1.0f / D) + eps);
    if (lane == 0 && WB_IN(row, 1, rows, SITE_STATS_OUT)) stats[row] = make_float2(mean, rstd);
    if (!AMAX) {
#pragma unroll
      for (int k = 0; k < NK; ++k) u[k] = nu[k];
      continue;
    }
    const int item = static_cast<int>(row / rows_per_item);
    if (item != run_item) {                        // rows are contiguous per warp: items change rarely
      flush();
      run_max2 = 0u;
      run_item = item;
    }
    const uint64_t nm2 = f32x2_pack(-mean, -mean), rs2 = f32x2_pack(rstd, rstd);
#pragma unroll
    for (int k = 0; k < NK; ++k) {
      const float4 g4 = __ldg(reinterpret_cast<const float4*>(g + 128 * k) + lane);
      const float4 b4 = __ldg(reinterpret_cast<const float4*>(bta + 128 * k) + lane);
      const uint32_t y01 = f32x2_to_bf16x2(
          ln_affine_x2(bf16x2_to_f32x2(u[k].x), nm2, rs2, f32x2_pack(g4.x, g4.y), f32x2_pack(b4.x, b4.y)));
      const uint32_t y23 = f32x2_to_bf16x2(
          ln_affine_x2(bf16x2_to_f32x2(u[k].y), nm2, rs2, f32x2_pack(g4.z, g4.w), f32x2_pack(b4.z, b4.w)));
      run_max2 = bf16x2_max(run_max2, bf16x2_max(y01 & 0x7fff7fffu, y23 & 0x7fff7fffu));
    }
#pragma unroll
    for (int k = 0; k < NK; ++k) u[k] = nu[k];
  }
  if (AMAX && r0 < r1) flush();
}

// Pass 2: q = E4M3 codes of bf16(LN(x)) scaled by 448 / amax[item] (1 if amax is 0), from the row
// statistics.  Column-stationary: a block spans one row, thread t owning columns 8t .. 8t+7 (gamma and
// beta in registers for every row it visits, one 16-byte load per row), and walks LNQ_ROWS consecutive
// rows, LNQ_RG loads in flight per thread.
constexpr int LNQ_RG = 8;
constexpr int LNQ_ROWS = 32;
__global__ void __launch_bounds__(256)
    ln_quantize_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ g,
                       const float* __restrict__ bta, const float2* __restrict__ stats, int rows, int d,
                       const float* __restrict__ amax, int rows_per_item, uint8_t* __restrict__ q) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int t = threadIdx.x;
  if (8 * t >= d) return;
  const int n_items = (rows + rows_per_item - 1) / rows_per_item;
  const float4 ga = __ldg(reinterpret_cast<const float4*>(g) + 2 * t), gb = __ldg(reinterpret_cast<const float4*>(g) + 2 * t + 1);
  const float4 ba = __ldg(reinterpret_cast<const float4*>(bta) + 2 * t), bb = __ldg(reinterpret_cast<const float4*>(bta) + 2 * t + 1);
  const uint64_t g2[4] = {f32x2_pack(ga.x, ga.y), f32x2_pack(ga.z, ga.w), f32x2_pack(gb.x, gb.y), f32x2_pack(gb.z, gb.w)};
  const uint64_t b2[4] = {f32x2_pack(ba.x, ba.y), f32x2_pack(ba.z, ba.w), f32x2_pack(bb.x, bb.y), f32x2_pack(bb.z, bb.w)};
  const int row0 = blockIdx.x * LNQ_ROWS;
  int item = row0 / rows_per_item;                 // items advance at most once every rows_per_item rows
  int item_end = (item + 1) * rows_per_item;
  float inv = 1.0f;
  if (WB_IN(item, 1, n_items, SITE_LNQ_AUX)) {
    const float a = __ldg(amax + item);
    inv = a > 0.0f ? 448.0f / a : 1.0f;
  }
  for (int rg = 0; rg < LNQ_ROWS; rg += LNQ_RG) {
    const int rb = row0 + rg;
    if (rb >= rows) break;
    uint4 u[LNQ_RG];
#pragma unroll
    for (int r = 0; r < LNQ_RG; ++r)
      u[r] = rb + r < rows && WB_IN(static_cast<long long>(rb + r) * d + 8 * t, 8, static_cast<long long>(rows) * d,
                                    SITE_LNQ_X)
                 ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<long long>(rb + r) * d) + t)
                 : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int r = 0; r < LNQ_RG; ++r) {
      const int row = rb + r;
      if (row >= rows) break;
      while (row >= item_end) {
        ++item;
        item_end += rows_per_item;
        const float a = WB_IN(item, 1, n_items, SITE_LNQ_AUX) ? __ldg(amax + item) : 0.0f;
        inv = a > 0.0f ? 448.0f / a : 1.0f;
      }
      const float2 st = WB_IN(row, 1, rows, SITE_LNQ_AUX) ? __ldg(stats + row) : make_float2(0.0f, 1.0f);
      const uint64_t nm2 = f32x2_pack(-st.x, -st.x), rs2 = f32x2_pack(st.y, st.y), inv2 = f32x2_pack(inv, inv);
      const uint32_t w[4] = {u[r].x, u[r].y, u[r].z, u[r].w};
      uint32_t c[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        float s0, s1, s2, s3;
        f32x2_unpack(f32x2_mul(bf16x2_to_f32x2(f32x2_to_bf16x2(ln_affine_x2(bf16x2_to_f32x2(w[2 * k]), nm2, rs2,
                                                                            g2[2 * k], b2[2 * k]))), inv2), s0, s1);
        f32x2_unpack(f32x2_mul(bf16x2_to_f32x2(f32x2_to_bf16x2(ln_affine_x2(bf16x2_to_f32x2(w[2 * k + 1]), nm2, rs2,
                                                                            g2[2 * k + 1], b2[2 * k + 1]))), inv2), s2, s3);
        c[k] = static_cast<uint32_t>(cvt_e4m3x2(s0, s1)) | (static_cast<uint32_t>(cvt_e4m3x2(s2, s3)) << 16);
      }
      if (WB_IN(static_cast<long long>(row) * d + 8 * t, 8, static_cast<long long>(rows) * d, SITE_LNQ_Q))
        reinterpret_cast<uint2*>(q + static_cast<long long>(row) * d)[t] = make_uint2(c[0], c[1]);
    }
  }
}

// ---------------------------------------------------------------------------
// LayerNorm folded into the following GEMM.  For y = LN(x; gamma, beta) W^T + b with
// LN(x) = (x - mean) rstd gamma + beta:
//   y[n] = rstd (sum_k x[k] W[n,k] gamma[k] - mean sum_k W[n,k] gamma[k]) + b[n] + sum_k beta[k] W[n,k],
// an identity of the LayerNorm definition.  The GEMM then reads x itself with B = W diag(gamma).
// ---------------------------------------------------------------------------

// (mean, rstd) of every row of x (bf16 [rows, d]) as LayerNorm computes them (two passes over the
// row in registers, rstd = 1 / sqrt(var + eps)); warp per row, 16-byte loads, no output rows.
constexpr int STATS_MAXC = 8;                  // 16-byte chunks per lane: d <= 8 * 32 * 8 = 2048
__global__ void ln_row_stats_kernel(const __nv_bfloat16* __restrict__ x, long long rows, int d, float eps,
                                    float2* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const long long warp_g = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int nc = d / 8;
  for (long long row = warp_g; row < rows; row += n_warps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + row * d);
    uint4 u[STATS_MAXC];
    float s1 = 0.0f;
#pragma unroll
    for (int i = 0; i < STATS_MAXC; ++i) {
      if (lane + 32 * i < nc && WB_IN(row * d + 8LL * (lane + 32 * i), 8, rows * d, SITE_ROWSTATS)) {
        u[i] = src[lane + 32 * i];
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u[i]);
#pragma unroll
        for (int j = 0; j < 8; ++j) s1 += __bfloat162float(h[j]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    const float mean = s1 / static_cast<float>(d);
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < STATS_MAXC; ++i) {
      if (lane + 32 * i < nc) {
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u[i]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float t = __bfloat162float(h[j]) - mean;
          q = fmaf(t, t, q);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    if (lane == 0 && WB_IN(row, 1, rows, SITE_ROWSTATS))
      out[row] = make_float2(mean, rsqrtf(q / static_cast<float>(d) + eps));
  }
}

// w_ln[n,k] = bf16(w[n,k] gamma[k]); c[n] = sum_k w_ln[n,k]; b_ln[n] = b[n] + sum_k beta[k] w[n,k].
// One warp per output row, lanes striding over k, fixed-order shuffle reduction (deterministic).
__global__ void fold_ln_kernel(const __nv_bfloat16* __restrict__ w, const float* __restrict__ b,
                               const float* __restrict__ gamma, const float* __restrict__ beta, int n_out, int d,
                               __nv_bfloat16* __restrict__ w_ln, float* __restrict__ c, float* __restrict__ b_ln) {
  const long long n = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (n >= n_out) return;
  const __nv_bfloat16* wr = w + n * d;
  __nv_bfloat16* orow = w_ln + n * d;
  float sc = 0.0f, sb = 0.0f;
  for (int k = lane; k < d; k += 32) {
    if (!WB_IN(n * d + k, 1, static_cast<long long>(n_out) * d, SITE_FOLD)) continue;
    const float wv = __bfloat162float(wr[k]);
    const __nv_bfloat16 f = __float2bfloat16_rn(wv * gamma[k]);
    orow[k] = f;
    sc += __bfloat162float(f);
    sb = fmaf(beta[k], wv, sb);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sc += __shfl_xor_sync(0xffffffffu, sc, o);
    sb += __shfl_xor_sync(0xffffffffu, sb, o);
  }
  if (lane == 0) {
    c[n] = sc;
    b_ln[n] = (b ? b[n] : 0.0f) + sb;
  }
}

// ---------------------------------------------------------------------------
// FP8 E4M3 per-tensor scaling.
// ---------------------------------------------------------------------------
__global__ void amax_kernel(const __nv_bfloat16* __restrict__ x, long long n, float* __restrict__ amax) {
  float m = 0.0f;
  const long long n8 = n / 8;
  const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = tid; i < n8; i += step) {
    if (!WB_IN(8 * i, 8, n, SITE_AMAX)) continue;
    uint4 u = reinterpret_cast<const uint4*>(x)[i];
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(__bfloat162float(h[j])));
  }
  for (long long i = n8 * 8 + tid; i < n; i += step) m = fmaxf(m, fabsf(__bfloat162float(x[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wm[32];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? wm[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0 && m > 0.0f) atomic_max_nonneg(amax, m);
  }
}

// code = E4M3_rn_satfinite(x * inv), inv = 448 / amax (1 if amax == 0), all float32.
__global__ void quantize_kernel(const __nv_bfloat16* __restrict__ x, long long n, uint8_t* __restrict__ q,
                                const float* __restrict__ amax, float* __restrict__ scale_out) {
  const float a = *amax;
  const float inv = a > 0.0f ? 448.0f / a : 1.0f;
  if (scale_out && blockIdx.x == 0 && threadIdx.x == 0) *scale_out = a > 0.0f ? a / 448.0f : 1.0f;
  const long long n16 = n / 16;
  const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = tid; i < n16; i += step) {
    if (!WB_IN(16 * i, 16, n, SITE_QUANT)) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x) + 2 * i;
    uint4 u0 = src[0], u1 = src[1];
    const __nv_bfloat16* h0 = reinterpret_cast<const __nv_bfloat16*>(&u0);
    const __nv_bfloat16* h1 = reinterpret_cast<const __nv_bfloat16*>(&u1);
    uint4 o;
    uint16_t* o16 = reinterpret_cast<uint16_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o16[j] = cvt_e4m3x2(__bfloat162float(h0[2 * j]) * inv, __bfloat162float(h0[2 * j + 1]) * inv);
      o16[4 + j] = cvt_e4m3x2(__bfloat162float(h1[2 * j]) * inv, __bfloat162float(h1[2 * j + 1]) * inv);
    }
    reinterpret_cast<uint4*>(q)[i] = o;
  }
  for (long long i = n16 * 16 + tid; i < n; i += step)
    q[i] = static_cast<uint8_t>(cvt_e4m3x2(__bfloat162float(x[i]) * inv, 0.0f) & 0xFF);
}

// Activation quantiser with one scale per batch item: rows of `cols` elements, item = row /
// rows_per_item, code = E4M3_rn_satfinite(x * inv_item), inv_item = 448 / amax[item] (1 if 0).
__global__ void quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, long long n, int cols, int rows_per_item,
                                     const float* __restrict__ amax, uint8_t* __restrict__ q) {
  const long long n16 = n / 16;
  const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long n_items = (n / cols + rows_per_item - 1) / rows_per_item;
  for (long long i = tid; i < n16; i += step) {
    const int item = static_cast<int>((i * 16) / cols / rows_per_item);
    if (!WB_IN(16 * i, 16, n, SITE_QUANT_ROWS) || !WB_IN(item, 1, n_items, SITE_QUANT_ROWS)) continue;
    const float a = __ldg(amax + item);
    const float inv = a > 0.0f ? 448.0f / a : 1.0f;
    const uint4* src = reinterpret_cast<const uint4*>(x) + 2 * i;
    uint4 u0 = src[0], u1 = src[1];
    const __nv_bfloat16* h0 = reinterpret_cast<const __nv_bfloat16*>(&u0);
    const __nv_bfloat16* h1 = reinterpret_cast<const __nv_bfloat16*>(&u1);
    uint4 o;
    uint16_t* o16 = reinterpret_cast<uint16_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o16[j] = cvt_e4m3x2(__bfloat162float(h0[2 * j]) * inv, __bfloat162float(h0[2 * j + 1]) * inv);
      o16[4 + j] = cvt_e4m3x2(__bfloat162float(h1[2 * j]) * inv, __bfloat162float(h1[2 * j + 1]) * inv);
    }
    reinterpret_cast<uint4*>(q)[i] = o;
  }
}

// E5M2 per-tensor cast: code = E5M2_rn_satfinite(x * 57344 / amax) (1 if amax == 0).
__global__ void quantize_e5m2_kernel(const __nv_bfloat16* __restrict__ x, long long n, uint8_t* __restrict__ q,
                                     const float* __restrict__ amax) {
  const float a = *amax;
  const float inv = a > 0.0f ? 57344.0f / a : 1.0f;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    uint16_t two;
    const float v = __bfloat162float(x[i]) * inv;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(two) : "f"(0.0f), "f"(v));
    q[i] = static_cast<uint8_t>(two & 0xFF);
  }
}

__global__ void finalize_scale_e5m2_kernel(float* p) {
  const float a = *p;
  *p = a > 0.0f ? a / 57344.0f : 1.0f;
}

__global__ void dequantize_e5m2_kernel(const uint8_t* __restrict__ q, const float* __restrict__ scale, long long n,
                                       __nv_bfloat16* __restrict__ y) {
  const float s = *scale;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint16_t two = static_cast<uint16_t>(q[i]);
    uint32_t h2;
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(two));
    y[i] = __float2bfloat16_rn(__half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFF))) * s);
  }
}

__global__ void finalize_scale_kernel(float* p) {
  const float a = *p;
  *p = a > 0.0f ? a / 448.0f : 1.0f;
}

__global__ void dequantize_kernel(const uint8_t* __restrict__ q, const float* __restrict__ scale, long long n,
                                  __nv_bfloat16* __restrict__ y) {
  const float s = *scale;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint16_t two = static_cast<uint16_t>(q[i]);
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
    const __half lo = __ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFF));
    y[i] = __float2bfloat16_rn(__half2float(lo) * s);
  }
}

// v [batch*T][ld] (head h at columns 64h..64h+63) -> f16 vt [(b*H + h)*64 + e][T_PAD]
static_assert(T_PAD % 8 == 0, "V^T rows are written in 8-position vectors");

// V [batch][T][ld] (bf16, head h in columns 64h .. 64h + 63) -> V^T [batch * H][64][T_PAD] (f16).
// A block moves a 128-position x 64-column tile of one head; each thread reads an 8 x 8 block as eight
// 16-byte row segments, transposes it in registers and writes eight 16-byte segments of V^T rows, so
// every global access is a full 16-byte vector (a warp's loads cover four 128-byte row segments).
// Positions T .. T_PAD - 1 of a V^T row are written as zeros.
__global__ void __launch_bounds__(128) transpose_v_kernel(const __nv_bfloat16* __restrict__ v, long long ld, int T,
                                                          int H, __half* __restrict__ vt) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int ty = threadIdx.x >> 3, cg = threadIdx.x & 7;    // 16 row groups x 8 column groups
  const int t0 = blockIdx.x * 128 + ty * 8;                  // first of this thread's 8 positions
  if (t0 >= T_PAD) return;
  const long long in_el = static_cast<long long>(gridDim.z) * T * ld;
  uint4 r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const long long vi = (static_cast<long long>(b) * T + t0 + i) * ld + h * 64 + cg * 8;
    r[i] = (t0 + i < T && WB_IN(vi, 8, in_el, SITE_TRANSPOSE_V_IN))
               ? *reinterpret_cast<const uint4*>(v + vi)
               : make_uint4(0u, 0u, 0u, 0u);
  }
  const long long out_el = static_cast<long long>(gridDim.z) * H * 64 * T_PAD;
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) {
    // column cg * 8 + jj of the eight rows: bf16 element jj of each row segment
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const uint32_t a = (&r[i].x)[jj >> 1], c = (&r[i + 1].x)[jj >> 1];
      const uint32_t ba = (jj & 1) ? (a >> 16) : (a & 0xffffu), bc = (jj & 1) ? (c >> 16) : (c & 0xffffu);
      const __half lo = __float2half_rn(__uint_as_float(ba << 16)), hi = __float2half_rn(__uint_as_float(bc << 16));
      w[i >> 1] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
    }
    const long long oi = (static_cast<long long>(b * H + h) * 64 + cg * 8 + jj) * T_PAD + t0;
    if (WB_IN(oi, 8, out_el, SITE_TRANSPOSE_V_OUT))
      *reinterpret_cast<uint4*>(vt + oi) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

// ------------------------------- launchers ---------------------------------
cudaError_t launch_pad_split(const float* audio, long long n_samples, long long stride, int n_chunks,
                             __nv_bfloat16* xs, cudaStream_t s) {
  pad_split_kernel<<<grid_for(static_cast<long long>(n_chunks) * PADDED, EW_THREADS), EW_THREADS, 0, s>>>(
      audio, n_samples, stride, n_chunks, xs);
  return cudaGetLastError();
}

cudaError_t launch_dft_basis(__nv_bfloat16* basis, cudaStream_t s) {
  dft_basis_kernel<<<(DFT_ROWS * N_FFT + 255) / 256, 256, 0, s>>>(basis);
  return cudaGetLastError();
}

cudaError_t launch_mel_fb(__nv_bfloat16* fbs, int n_mels, cudaStream_t s) {
  mel_fb_kernel<<<(MEL_ROWS * N_BIN_PAD + 255) / 256, 256, 0, s>>>(fbs, n_mels);
  return cudaGetLastError();
}

cudaError_t launch_logmel_post(float* out, const float* mel_max, int n_chunks, int n_mels, cudaStream_t s) {
  const int per_chunk = n_mels * N_FRAMES;
  dim3 grid(grid_for(per_chunk / 4, EW_THREADS, 64), n_chunks);
  logmel_post_kernel<<<grid, EW_THREADS, 0, s>>>(out, mel_max, per_chunk);
  return cudaGetLastError();
}

cudaError_t launch_stem_transpose(const float* logmel, int batch, int n_mels, __nv_bfloat16* yTp,
                                  cudaStream_t s) {
  dim3 grid((N_FRAMES + 31) / 32, (n_mels + 31) / 32, batch);
  stem_transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(logmel, n_mels, yTp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_zero_rows(yTp, n_mels, static_cast<long long>(N_FRAMES + 2) * n_mels, batch, 0, s);
  if (e != cudaSuccess) return e;
  return launch_zero_rows(yTp, n_mels, static_cast<long long>(N_FRAMES + 2) * n_mels, batch, N_FRAMES + 1, s);
}

cudaError_t launch_zero_rows(__nv_bfloat16* base, long long row_elems, long long batch_stride_elems, int batch,
                             int row, cudaStream_t s) {
  dim3 grid(grid_for(row_elems, EW_THREADS, 16), batch);
  zero_rows_kernel<<<grid, EW_THREADS, 0, s>>>(base, row_elems, batch_stride_elems, batch, row);
  return cudaGetLastError();
}

cudaError_t launch_pack_conv(const float* w, int c_out, int c_in, __nv_bfloat16* packed, cudaStream_t s) {
  pack_conv_kernel<<<grid_for(static_cast<long long>(c_out) * c_in * 3, EW_THREADS), EW_THREADS, 0, s>>>(
      w, c_out, c_in, packed);
  return cudaGetLastError();
}

template <int NV, int VEC, bool RMS>
static cudaError_t ln_launch(const __nv_bfloat16* x, const __nv_bfloat16* res, const float* g, const float* b,
                             int rows, float eps, __nv_bfloat16* y, __nv_bfloat16* total, cudaStream_t s) {
  // persistent grid: 2 blocks of 8 warps per SM, each warp walking a contiguous range of rows
  long long blocks = (rows + LN_WARPS - 1) / LN_WARPS;
  const long long cap = 2LL * sm_count();
  if (blocks > cap) blocks = cap;
  if (res)
    layernorm_kernel<NV, VEC, true, RMS><<<static_cast<int>(blocks), LN_WARPS * 32, 0, s>>>(
        x, res, g, b, rows, eps, y, total);
  else
    layernorm_kernel<NV, VEC, false, RMS><<<static_cast<int>(blocks), LN_WARPS * 32, 0, s>>>(
        x, res, g, b, rows, eps, y, total);
  return cudaGetLastError();
}

template <bool RMS>
static cudaError_t norm_dispatch(const __nv_bfloat16* x, const __nv_bfloat16* res, const float* g, const float* b,
                                 int rows, int d, float eps, __nv_bfloat16* y, __nv_bfloat16* total, cudaStream_t s) {
#define WB_LN_CASE(NV, VEC) \
  case NV * VEC * 32:       \
    return ln_launch<NV, VEC, RMS>(x, res, g, b, rows, eps, y, total, s);
  switch (d) {
    WB_LN_CASE(1, 4)
    WB_LN_CASE(1, 8)
    WB_LN_CASE(3, 4)
    WB_LN_CASE(2, 8)
    WB_LN_CASE(5, 4)
    WB_LN_CASE(3, 8)
    WB_LN_CASE(7, 4)
    WB_LN_CASE(4, 8)
    WB_LN_CASE(9, 4)
    WB_LN_CASE(5, 8)
    WB_LN_CASE(11, 4)
    WB_LN_CASE(6, 8)
    WB_LN_CASE(13, 4)
    WB_LN_CASE(7, 8)
    WB_LN_CASE(15, 4)
    WB_LN_CASE(8, 8)
    default:
      return cudaErrorInvalidValue;
  }
#undef WB_LN_CASE
}

template <int NK>
static cudaError_t ln_e4m3_launch(const __nv_bfloat16* x, const float* g, const float* b, int rows, float eps,
                                  float2* stats, float* amax, int rows_per_item, uint8_t* q, cudaStream_t s) {
  constexpr int D = NK * 128;
  long long blocks = (rows + LN_WARPS - 1) / LN_WARPS;
  const long long cap = 2LL * sm_count();
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_pdl(ln_stats_amax_kernel<NK, true>, dim3(static_cast<unsigned>(blocks)), dim3(LN_WARPS * 32), 0,
                             s, x, g, b, rows, eps, stats, amax, rows_per_item);
  if (e != cudaSuccess) return e;
  const int threads = ((D / 8 + 31) / 32) * 32;
  return launch_pdl(ln_quantize_kernel, dim3((rows + LNQ_ROWS - 1) / LNQ_ROWS), dim3(threads), 0, s, x, g, b,
                    static_cast<const float2*>(stats), rows, D, static_cast<const float*>(amax), rows_per_item, q);
}

cudaError_t launch_layernorm_e4m3(const __nv_bfloat16* x, const float* g, const float* b, int rows, int d, float eps,
                                  float2* stats, float* amax, int rows_per_item, uint8_t* q, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int rpi = rows_per_item > 0 ? rows_per_item : rows;
  switch (d) {
    case 128: return ln_e4m3_launch<1>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 256: return ln_e4m3_launch<2>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 384: return ln_e4m3_launch<3>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 512: return ln_e4m3_launch<4>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 640: return ln_e4m3_launch<5>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 768: return ln_e4m3_launch<6>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 896: return ln_e4m3_launch<7>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 1024: return ln_e4m3_launch<8>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 1152: return ln_e4m3_launch<9>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 1280: return ln_e4m3_launch<10>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 1408: return ln_e4m3_launch<11>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 1536: return ln_e4m3_launch<12>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 1664: return ln_e4m3_launch<13>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 1792: return ln_e4m3_launch<14>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 1920: return ln_e4m3_launch<15>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    case 2048: return ln_e4m3_launch<16>(x, g, b, rows, eps, stats, amax, rpi, q, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_layernorm(const __nv_bfloat16* x, const __nv_bfloat16* res, const float* g, const float* b,
                             int rows, int d, float eps, __nv_bfloat16* y, __nv_bfloat16* total, cudaStream_t s) {
  return norm_dispatch<false>(x, res, g, b, rows, d, eps, y, total, s);
}

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* res, const float* g, int rows, int d,
                           float eps, __nv_bfloat16* y, __nv_bfloat16* total, cudaStream_t s) {
  return norm_dispatch<true>(x, res, g, nullptr, rows, d, eps, y, total, s);
}

template <int NK>
static cudaError_t ln_stats_launch(const __nv_bfloat16* x, int rows, float eps, float2* out, cudaStream_t s) {
  long long blocks = (rows + LN_WARPS - 1) / LN_WARPS;
  const long long cap = 3LL * sm_count();   // 80 registers: three blocks of eight warps fit an SM
  if (blocks > cap) blocks = cap;
  return launch_pdl(ln_stats_amax_kernel<NK, false>, dim3(static_cast<unsigned>(blocks)), dim3(LN_WARPS * 32), 0, s, x,
                    static_cast<const float*>(nullptr), static_cast<const float*>(nullptr), rows, eps, out,
                    static_cast<float*>(nullptr), 1);
}

// (mean, rstd) of each row from the (mean, M2) of its n_groups column groups of `group` values each,
// stored group-major (part[g * rows + r]) as the residual GEMM epilogues leave them, merged about the
// first group's mean (the pairwise update of Chan, Golub and LeVeque for equal counts).  A block
// takes 32 rows: warp w sums the groups w, w + 8, .. of the 32 rows (each load 256 contiguous bytes)
// and shared memory adds the eight warps' sums.
constexpr int MERGE_SLICES = 8;
__global__ void __launch_bounds__(32 * MERGE_SLICES) ln_merge_kernel(const float2* __restrict__ part, int rows,
                                                                     int n_groups, int group, float eps,
                                                                     float2* __restrict__ stats) {
  __shared__ float red[3][MERGE_SLICES][33];
  grid_dependency_wait();
  grid_dependents_launch();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long long row = static_cast<long long>(blockIdx.x) * 32 + lane;
  const long long n_el = static_cast<long long>(rows) * n_groups;
  float s1 = 0.0f, s2 = 0.0f, s3 = 0.0f, m0 = 0.0f;
  if (row < rows) {
    m0 = WB_IN(row, 1, n_el, SITE_LNMERGE_IN) ? part[row].x : 0.0f;
    for (int gi = w; gi < n_groups; gi += MERGE_SLICES) {
      const long long i = static_cast<long long>(gi) * rows + row;
      if (!WB_IN(i, 1, n_el, SITE_LNMERGE_IN)) continue;
      const float2 t = part[i];
      const float dl = t.x - m0;
      s1 += dl;
      s2 = fmaf(dl, dl, s2);
      s3 += t.y;
    }
  }
  red[0][w][lane] = s1;
  red[1][w][lane] = s2;
  red[2][w][lane] = s3;
  __syncthreads();
  if (w != 0 || row >= rows) return;
  s1 = s2 = s3 = 0.0f;
#pragma unroll
  for (int k = 0; k < MERGE_SLICES; ++k) {
    s1 += red[0][k][lane];
    s2 += red[1][k][lane];
    s3 += red[2][k][lane];
  }
  if (WB_IN(row, 1, rows, SITE_LNMERGE_OUT)) {
    const float ng = static_cast<float>(n_groups);
    const float m2 = s3 + static_cast<float>(group) * fmaxf(s2 - s1 * s1 / ng, 0.0f);
    stats[row] = make_float2(m0 + s1 / ng, rsqrtf(m2 / (ng * static_cast<float>(group)) + eps));
  }
}

cudaError_t launch_ln_merge(const float2* part, long long rows, int n_groups, int group, float eps, float2* out,
                            cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (rows >= (1LL << 31) || n_groups < 1 || group < 1) return cudaErrorInvalidValue;
  return launch_pdl(ln_merge_kernel, dim3(static_cast<unsigned>((rows + 31) / 32)), dim3(32 * MERGE_SLICES), 0, s,
                    part, static_cast<int>(rows), n_groups, group, eps, out);
}

cudaError_t launch_ln_stats(const __nv_bfloat16* x, long long rows, int d, float eps, float2* out, cudaStream_t s) {
  // widths that are multiples of 128 (every Whisper size): the persistent row walk
  if (rows > 0 && rows < (1LL << 31)) {
    const int r = static_cast<int>(rows);
    switch (d) {
      case 384: return ln_stats_launch<3>(x, r, eps, out, s);
      case 512: return ln_stats_launch<4>(x, r, eps, out, s);
      case 768: return ln_stats_launch<6>(x, r, eps, out, s);
      case 1024: return ln_stats_launch<8>(x, r, eps, out, s);
      case 1280: return ln_stats_launch<10>(x, r, eps, out, s);
      default: break;
    }
  }
  if (d <= 0 || d % 8 || d > STATS_MAXC * 32 * 8) return cudaErrorInvalidValue;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;               // 8 warps per block, a warp per row
  ln_row_stats_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(x, rows, d, eps, out);
  return cudaGetLastError();
}

cudaError_t launch_fold_ln(const __nv_bfloat16* w, const float* b, const float* gamma, const float* beta, int n_out,
                           int d, __nv_bfloat16* w_ln, float* c, float* b_ln, cudaStream_t s) {
  const long long threads = static_cast<long long>(n_out) * 32;
  if (threads == 0) return cudaSuccess;
  fold_ln_kernel<<<static_cast<int>((threads + 255) / 256), 256, 0, s>>>(w, b, gamma, beta, n_out, d, w_ln, c, b_ln);
  return cudaGetLastError();
}

cudaError_t launch_amax(const __nv_bfloat16* x, long long n, float* amax, cudaStream_t s) {
  amax_kernel<<<grid_for(n / 8 + 1, EW_THREADS, 152 * 8), EW_THREADS, 0, s>>>(x, n, amax);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const __nv_bfloat16* x, long long n, uint8_t* q, const float* amax, float* scale_out,
                            cudaStream_t s) {
  quantize_kernel<<<grid_for(n / 16 + 1, EW_THREADS, 152 * 16), EW_THREADS, 0, s>>>(x, n, q, amax, scale_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const __nv_bfloat16* x, long long n, int cols, int rows_per_item,
                                 const float* amax, uint8_t* q, cudaStream_t s) {
  quantize_rows_kernel<<<grid_for(n / 16 + 1, EW_THREADS, 152 * 16), EW_THREADS, 0, s>>>(x, n, cols, rows_per_item,
                                                                                        amax, q);
  return cudaGetLastError();
}

cudaError_t launch_finalize_scale(float* amax_to_scale, cudaStream_t s) {
  finalize_scale_kernel<<<1, 1, 0, s>>>(amax_to_scale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e5m2(const __nv_bfloat16* x, long long n, uint8_t* q, float* amax_to_scale,
                                 cudaStream_t s) {
  quantize_e5m2_kernel<<<grid_for(n, EW_THREADS), EW_THREADS, 0, s>>>(x, n, q, amax_to_scale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  finalize_scale_e5m2_kernel<<<1, 1, 0, s>>>(amax_to_scale);
  return cudaGetLastError();
}

cudaError_t launch_dequantize_e5m2(const uint8_t* q, const float* scale, long long n, __nv_bfloat16* y,
                                   cudaStream_t s) {
  dequantize_e5m2_kernel<<<grid_for(n, EW_THREADS), EW_THREADS, 0, s>>>(q, scale, n, y);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* q, const float* scale, long long n, __nv_bfloat16* y,
                              cudaStream_t s) {
  dequantize_kernel<<<grid_for(n, EW_THREADS), EW_THREADS, 0, s>>>(q, scale, n, y);
  return cudaGetLastError();
}

cudaError_t launch_transpose_v(const __nv_bfloat16* v, long long ld, int batch, int T, int H, __half* vt,
                               cudaStream_t s) {
  dim3 grid((T_PAD + 127) / 128, H, batch);
  transpose_v_kernel<<<grid, 128, 0, s>>>(v, ld, T, H, vt);
  return cudaGetLastError();
}

// pos[t][n] = sinusoid(t, n, d): the conv stem's position table, [T][d] float32.
__global__ void pos_table_kernel(float* __restrict__ pos, int T, int d) {
  const long long n_el = static_cast<long long>(T) * d;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n_el; i += step)
    pos[i] = sinusoid(static_cast<int>(i / d), static_cast<int>(i % d), d);
}

cudaError_t launch_pos_table(float* pos, int T, int d, cudaStream_t s) {
  pos_table_kernel<<<grid_for(static_cast<long long>(T) * d, EW_THREADS), EW_THREADS, 0, s>>>(pos, T, d);
  return cudaGetLastError();
}

// Diagnostic of the bounded-wait path: one thread waits on an mbarrier that
// nothing ever arrives on.  mbar_wait gives up after its time limit, records
// ERR_TIMEOUT with the site in the device error word and the kernel returns
// normally, exactly as a stalled pipeline role would.
__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint32_t site) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_wait(&bar, 0, err, &abort_flag, site);
}

cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint32_t site, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err, site);
  return cudaGetLastError();
}

// Diagnostic of the debug bounds checks: evaluates one check on an index outside the stated extent
// (11 of 10 elements).  Nothing is read or written but the error word: a debug build records
// ERR_BOUNDS with the site, a release build compiles the check away and records nothing.
__global__ void bounds_check_selftest_kernel(uint32_t site) {
  if (threadIdx.x == 0 && blockIdx.x == 0) (void)in_bounds(&g_simt_err, 10, 1, 10, site);
}

cudaError_t launch_bounds_check_selftest(uint32_t site, cudaStream_t s) {
  bounds_check_selftest_kernel<<<1, 32, 0, s>>>(site);
  return cudaGetLastError();
}

uint32_t* simt_err_ptr() {
  constexpr int kMaxDev = 64;
  static uint32_t* ptrs[kMaxDev] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_simt_err) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

}  // namespace wb
