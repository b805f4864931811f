// Host-side declarations shared by the translation units of libwb.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "types.h"

namespace wb {

constexpr int N_FFT = 400;
constexpr int HOP = 160;
constexpr int N_FRAMES = 3000;
constexpr int CHUNK = 480000;
constexpr int PAD = N_FFT / 2;
constexpr int PADDED = CHUNK + 2 * PAD;      // 480400 samples per reflect-padded chunk
constexpr int DFT_ROWS = 512;                // 2 tiles x (128 cos + 128 sin) basis rows
constexpr int N_BIN_PAD = 256;               // power-spectrum bins padded 201 -> 256
constexpr int MEL_ROWS = 128;                // mel filterbank rows padded to one N tile
constexpr int T_TOK = 1500;                  // encoder positions per chunk
constexpr int T_PAD = 1504;                  // V^T row length (16-byte aligned rows)

// ---- launchers of the SIMT kernels (kernels.cu) ----
cudaError_t launch_pad_split(const float* audio, long long n_samples, long long stride, int n_chunks,
                             __nv_bfloat16* xs, cudaStream_t s);
cudaError_t launch_dft_basis(__nv_bfloat16* basis, cudaStream_t s);
cudaError_t launch_mel_fb(__nv_bfloat16* fbs, int n_mels, cudaStream_t s);
cudaError_t launch_logmel_post(float* out, const float* mel_max, int n_chunks, int n_mels, cudaStream_t s);
cudaError_t launch_stem_transpose(const float* logmel, int batch, int n_mels, __nv_bfloat16* yTp,
                                  cudaStream_t s);
cudaError_t launch_pack_conv(const float* w, int c_out, int c_in, __nv_bfloat16* packed, cudaStream_t s);
cudaError_t launch_layernorm(const __nv_bfloat16* x, const __nv_bfloat16* res, const float* g, const float* b,
                             int rows, int d, float eps, __nv_bfloat16* y, __nv_bfloat16* total, cudaStream_t s);
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* res, const float* g, int rows, int d,
                           float eps, __nv_bfloat16* y, __nv_bfloat16* total, cudaStream_t s);
// LayerNorm to E4M3 codes in two passes (row statistics + per-item absmax, then codes); the same
// widths as launch_layernorm (multiples of 128 up to 2048).
cudaError_t launch_layernorm_e4m3(const __nv_bfloat16* x, const float* g, const float* b, int rows, int d, float eps,
                                  float2* stats, float* amax, int rows_per_item, uint8_t* q, cudaStream_t s);
cudaError_t launch_ln_stats(const __nv_bfloat16* x, long long rows, int d, float eps, float2* out, cudaStream_t s);
cudaError_t launch_ln_merge(const float2* part, long long rows, int n_groups, int group, float eps, float2* out,
                            cudaStream_t s);
cudaError_t launch_fold_ln(const __nv_bfloat16* w, const float* b, const float* gamma, const float* beta, int n_out,
                           int d, __nv_bfloat16* w_ln, float* c, float* b_ln, cudaStream_t s);
cudaError_t launch_quantize_e5m2(const __nv_bfloat16* x, long long n, uint8_t* q, float* amax_to_scale,
                                 cudaStream_t s);
cudaError_t launch_dequantize_e5m2(const uint8_t* q, const float* scale, long long n, __nv_bfloat16* y,
                                   cudaStream_t s);
cudaError_t launch_quantize_rows(const __nv_bfloat16* x, long long n, int cols, int rows_per_item,
                                 const float* amax, uint8_t* q, cudaStream_t s);
cudaError_t launch_amax(const __nv_bfloat16* x, long long n, float* amax, cudaStream_t s);
cudaError_t launch_quantize(const __nv_bfloat16* x, long long n, uint8_t* q, const float* amax,
                            float* scale_out, cudaStream_t s);
cudaError_t launch_finalize_scale(float* amax_to_scale, cudaStream_t s);
cudaError_t launch_dequantize(const uint8_t* q, const float* scale, long long n, __nv_bfloat16* y,
                              cudaStream_t s);
cudaError_t launch_transpose_v(const __nv_bfloat16* v, long long ld, int batch, int T, int H, __half* vt,
                               cudaStream_t s);
cudaError_t launch_zero_rows(__nv_bfloat16* base, long long row_elems, long long batch_stride_elems,
                             int batch, int row, cudaStream_t s);
cudaError_t launch_pos_table(float* pos, int T, int d, cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint32_t site, cudaStream_t s);
cudaError_t launch_bounds_check_selftest(uint32_t site, cudaStream_t s);
// Device address of the error word of the SIMT kernels' debug bounds checks (per device, looked up
// once); null if it cannot be found.
uint32_t* simt_err_ptr();

// Launch with programmatic stream serialization: the kernel may begin (its prologue, up to its
// grid_dependency_wait()) while the previous kernel in the stream is still finishing.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---- tensor-core kernels (tc_kernels.cu) ----
struct GemmLaunch {
  CUtensorMap amap[GEMM_MAX_AMAPS];
  CUtensorMap bmap;
  CUtensorMap omap;   // output boxes (32 x 32 bf16, 64-byte swizzle), standard epilogues only
  GemmParams p;
  int bn;       // 128 or 256
  bool fp8;
  int epi;      // EpiKind
};
cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t s);
cudaError_t launch_attention(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& vt,
                             const AttnParams& p, cudaStream_t s);
int sm_count();

}  // namespace wb
