// Plain data types and constants shared by the host launch code and the
// tensor-core kernels (no device code here).
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace wb {

// Bits of the device error word (bits 8..15 carry the site of a timed-out wait).
enum : uint32_t { ERR_TIMEOUT = 1u, ERR_BOUNDS = 2u };

constexpr int GEMM_BM = 128;
constexpr int GEMM_THREADS = 192;
constexpr int GEMM_MAX_PASSES = 24;
constexpr int GEMM_MAX_AMAPS = 4;

enum EpiKind : int { EPI_STD = 0, EPI_POWER = 1, EPI_MEL = 2 };

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
  // ---- standard epilogue: y = act(alpha * acc + bias) (+ pe) (+ resid) ----
  void* out;                 // bf16 output
  long long ldo;             // elements between output rows
  long long out_batch_rows;  // output rows between batch items
  int out_row_off;           // extra row offset inside a batch item
  const float* bias;         // [N] or null
  const float* scale_a;      // device scalars multiplied into alpha (E4M3 operand scales) or null
  const float* scale_b;
  int act_gelu;              // 1: exact-erf GELU after the bias
  int add_pe;                // 1: add the sinusoidal position table (row = position, col = channel)
  const __nv_bfloat16* resid;  // residual added last, same indexing as out, or null
  float* amax;               // if set: atomic max of |y| (feeds a per-tensor E4M3 scale)
  // QKV: columns >= vt_col0 are written transposed to vt[(b*H + h)*64 + e][t]
  __nv_bfloat16* vt;
  int vt_col0, vt_T, vt_ld;  // tokens per batch item, elements between vt rows
  // ---- DFT power epilogue: P split into hi/lo bf16 parts ----
  __nv_bfloat16* pw;         // [batch][2][M][pw_ld]
  int pw_ld;
  // ---- mel epilogue: log10 written as [batch][n_valid][M] + per-item max ----
  float* mel_out;
  float* mel_max;            // [batch] max of the mel power (bit pattern, >= 0)
  int n_valid;
  uint32_t* err;
};

constexpr int ATT_BQ = 128;
constexpr int ATT_BKV = 128;
constexpr int ATT_HD = 64;
constexpr int ATT_STAGES = 3;
constexpr int ATT_THREADS = 192;

struct AttnSmem {
  static constexpr int Q_BYTES = ATT_BQ * 128;        // [128 q][64 e] bf16
  static constexpr int K_BYTES = ATT_BKV * 128;       // [128 kv][64 e]
  static constexpr int V_BYTES = 2 * ATT_HD * 128;    // 2 halves of [64 e][64 kv]
  static constexpr int P_BYTES = 2 * ATT_BQ * 128;    // 2 halves of [128 q][64 kv]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + ATT_STAGES * K_BYTES;
  static constexpr int OFF_P = OFF_V + ATT_STAGES * V_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int TOTAL = 1024 + OFF_BAR + 256;
};

struct AttnParams {
  int T;            // sequence length (1500)
  int H;            // heads
  int d;            // model width = H * 64
  int batch;
  float scale_log2; // log2(e) / sqrt(64)
  __nv_bfloat16* out;  // [batch * T, d]
  uint32_t* err;
};

}  // namespace wb
