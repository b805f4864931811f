// Plain data types and constants shared by the host launch code and the
// tensor-core kernels (no device code here).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace wb {

// Bits of the device error word (bits 8..15 carry the site of a timed-out wait).
enum : uint32_t { ERR_TIMEOUT = 1u, ERR_BOUNDS = 2u };

constexpr int GEMM_BM = 128;
constexpr int GEMM_EPI_WARPS = 16;                      // 4 per TMEM lane quarter
constexpr int GEMM_THREADS = 64 + 32 * GEMM_EPI_WARPS;   // producer + MMA + epilogue warps
constexpr int GEMM_MAX_PASSES = 24;
constexpr int GEMM_MAX_AMAPS = 4;

// Epilogue kinds (compile-time): what happens to each fp32 accumulator after the mainloop.
enum EpiKind : int {
  EPI_BIAS = 0,        // y = alpha*acc + bias                     (QKV with the V^T side output, plain linear)
  EPI_BIAS_GELU = 1,   // y = GELU(alpha*acc + bias)               (FC1, conv1)
  EPI_BIAS_RESID = 2,  // y = [GELU](alpha*acc + bias) + resid     (out-proj, FC2)
  EPI_CONV2 = 3,       // y = GELU(acc + bias) + pos[row][col] (conv2, sinusoidal position table)
  EPI_POWER = 4,       // DFT: |X|^2 split into bf16 hi/lo parts
  EPI_MEL = 5          // mel: log10(max(acc, 1e-10)) written transposed, per-item max
};

struct GemmPass {
  int8_t amap, a_part, a_row_off, b_part;
  int16_t a_x0, b_x0;
  int16_t n_kb, pad;
};

struct GemmParams {
  int M;             // output rows per batch item
  int N;             // output columns (multiple of 32)
  int batch;         // batch items (A's 4th tensor-map coordinate)
  int n_pass;
  GemmPass pass[GEMM_MAX_PASSES];
  // ---- standard epilogues: the output (and residual) tiles move through TMA maps ----
  int out_row_off;           // row offset of row 0 of an item inside the output map
  const float* bias;         // [N] or null
  const float* scale_a;      // device scalars multiplied into alpha (E4M3 operand scales) or null
  const float* scale_b;
  const float* amax_a;       // if set: per-item absmax of the E4M3 A operand; row m of item i is
                             // scaled by (amax_a[i] > 0 ? amax_a[i] / 448 : 1) instead of *scale_a
  int rows_per_item;         // rows of one batch item (chunk) in the flattened row index
  int act_gelu;              // EPI_BIAS_RESID only: GELU before the residual add
  const __nv_bfloat16* resid;  // EPI_BIAS_RESID: residual, element (item, row, n) at
  long long resid_ld;          //   resid[item * resid_item + (out_row_off + row) * resid_ld + n]
  long long resid_item;
  // EPI_BIAS / EPI_BIAS_GELU, bf16: a LayerNorm folded into this GEMM.  A is the un-normalised row x,
  // B = W diag(gamma), ln_stats[r] = (mean, rstd) of flattened row r = b*M + m, and the epilogue
  // forms rstd (acc - mean ln_c[n]) + bias[n]
  const float2* ln_stats;
  const float* ln_c;
  // EPI_BIAS_RESID: if set, per output row r (of batch * M) and 32-column group g,
  // ln_part[g * batch * M + r] = (mean, M2) of the group's stored (bf16) values: the next
  // LayerNorm's statistics, before merging
  float2* ln_part;
  float* amax;               // if set: per-item atomic max of |y| (feeds the next E4M3 operand's scale)
  const float* pos;          // EPI_CONV2: position table [M][N] (float32), added after the GELU
  // QKV: columns >= vt_col0 are written transposed, as f16, to vt[(b*H + h)*64 + e][t]
  __half* vt;
  int vt_col0, vt_T, vt_ld;  // tokens per batch item, elements between vt rows
  // ---- DFT power epilogue: P split into hi/lo bf16 parts ----
  __nv_bfloat16* pw;         // [batch][2][M][pw_ld]
  int pw_ld;
  // ---- mel epilogue: log10 written as [batch][n_valid][M] + per-item max ----
  float* mel_out;
  float* mel_max;            // [batch] max of the mel power (bit pattern, >= 0)
  int n_valid;
  uint32_t* err;
  // extents (elements) of the buffers the epilogue reaches with plain loads and stores, for the
  // bounds checks of debug builds (unused otherwise)
  long long resid_elems, vt_elems, pw_elems, mel_elems;
  int amax_items;            // entries of amax / amax_a
};

constexpr int ATT_BQ = 128;           // queries per CTA
constexpr int ATT_BKV = 128;          // keys per step
constexpr int ATT_HD = 64;            // head dim
constexpr int ATT_KSTAGES = 3;        // K tiles in flight
constexpr int ATT_VSTAGES = 2;        // V^T tiles in flight
constexpr int ATT_SOFTMAX_WARPS = 8;  // two per TMEM lane quarter, 16 query rows each
constexpr int ATT_THREADS = 64 + 32 * ATT_SOFTMAX_WARPS;   // producer + MMA + softmax warps
constexpr int ATT_CTAS_PER_SM = 2;
// TMEM columns of one CTA (two CTAs share the 512 of an SM): S (128 fp32), O (64 fp32),
// P (128 keys as 64 packed f16 columns).
constexpr uint32_t ATT_TM_S = 0, ATT_TM_O = 128, ATT_TM_P = 192, ATT_TM_COLS = 256;

struct AttnSmem {
  static constexpr int Q_BYTES = ATT_BQ * 128;              // [128 q][64 e] bf16
  static constexpr int K_BYTES = ATT_BKV * 128;             // [128 kv][64 e] bf16
  static constexpr int VH_BYTES = ATT_HD * 128;             // one V^T half: [64 e][64 kv] f16
  static constexpr int V_BYTES = 2 * VH_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + ATT_KSTAGES * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + ATT_VSTAGES * V_BYTES;
  static constexpr int TOTAL = 1024 + OFF_BAR + 256;
};
static_assert(2 * AttnSmem::TOTAL <= 227 * 1024, "two attention CTAs must fit one SM");

struct AttnParams {
  int T;            // sequence length (1500)
  int H;            // heads
  int d;            // model width = H * 64
  int batch;
  float scale_log2; // log2(e) / sqrt(64)
  __nv_bfloat16* out;  // [batch * T, d]
  float* amax;         // if set: amax[b] = max |bf16 output| over batch item b (atomic; for an E4M3 scale)
  uint32_t* err;
};

// Sites (bits 8..15 of the error word) of the debug bounds checks: 0x20-0x3F the SIMT kernels,
// 0x40-0x4F the GEMM epilogues, 0x50-0x5F the attention epilogue.
enum : uint32_t {
  SITE_PAD_SPLIT = 0x20, SITE_DFT_BASIS, SITE_MEL_FB, SITE_LOGMEL_POST, SITE_STEM_T_IN, SITE_STEM_T_OUT,
  SITE_ZERO_ROWS, SITE_PACK_CONV, SITE_LN_X, SITE_LN_Y, SITE_LN_GB, SITE_STATS_X, SITE_STATS_OUT,
  SITE_STATS_AMAX, SITE_LNQ_X, SITE_LNQ_Q, SITE_LNQ_AUX, SITE_ROWSTATS, SITE_FOLD, SITE_QUANT,
  SITE_QUANT_ROWS, SITE_E5M2, SITE_DEQUANT, SITE_TRANSPOSE_V_IN, SITE_TRANSPOSE_V_OUT, SITE_POS, SITE_AMAX,
  SITE_LNMERGE_IN, SITE_LNMERGE_OUT,
  SITE_GEMM_RESID = 0x40, SITE_GEMM_BIAS, SITE_GEMM_LNSTATS, SITE_GEMM_POS, SITE_GEMM_VT, SITE_GEMM_POWER,
  SITE_GEMM_MEL, SITE_GEMM_AMAX, SITE_GEMM_LNPART,
  SITE_ATT_OUT = 0x50, SITE_ATT_AMAX
};

}  // namespace wb
