/*
 * wb.h - C ABI of libwb, the GB300 (sm_103a) hot path of batched Whisper
 * large-v3 encoding: float32 16 kHz audio -> log-mel -> conv stem -> encoder
 * hidden states, with a per-layer-site precision choice (bf16 or FP8 E4M3).
 *
 * Conventions shared by every entry point
 *  - All tensor arguments are DEVICE pointers owned by the caller; libwb never
 *    allocates or frees memory.  Scratch memory is passed in as a workspace
 *    whose size the matching *_workspace_bytes() query returns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and stream-ordered with the caller's other work.
 *  - Argument errors are detected on the host before anything is launched and
 *    returned synchronously (WB_EINVAL, WB_EUNSUPPORTED, WB_EWORKSPACE).
 *    Launch failures return WB_ECUDA.  Faults found on the device (a bounded
 *    wait that ran out) are recorded in a device error word and reported by
 *    wb_check_device_error().  No kernel traps.
 *  - Pointers must be 16-byte aligned.  bf16 tensors hold IEEE bfloat16 bit
 *    patterns; E4M3 tensors hold OCP FP8 E4M3 ("fn") codes.
 *  - Row-major layouts throughout; "[a, b]" means b is contiguous.
 *  - libwb looks up a few device addresses of its own (the device error word,
 *    the scratch array of wb_logmel_static) once per device and keeps them;
 *    cudaDeviceReset() invalidates them, so a process must not call libwb on
 *    a device after resetting it.
 *
 * Sources (the pages this library follows): the whisper-blaze PyPI page
 * ("Quick Start", "Batch Transcription", "Direct Kernel API") and the
 * whisper-blaze showcase site ("The Approach", "The Solution", "Learnings").
 */
#ifndef WB_H
#define WB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WB_OK = 0,
  WB_EINVAL = -1,        /* bad pointer, size or layout argument */
  WB_ECUDA = -2,         /* a CUDA runtime/driver call or launch failed */
  WB_EUNSUPPORTED = -3,  /* valid request this library does not implement (e.g. mixed bf16 x E4M3 site) */
  WB_ETIMEOUT = -4,      /* a bounded device-side wait ran out (reported by wb_check_device_error) */
  WB_EWORKSPACE = -5,    /* workspace pointer null or smaller than the *_workspace_bytes() query */
  WB_EBOUNDS = -6        /* debug builds only: a kernel index fell outside its buffer (wb_check_device_error) */
} wb_status;

/* Element types of one precision site (showcase site, "The Approach": a
 * PrecisionConfig assigns weight and activation precision per layer site). */
typedef enum { WB_BF16 = 0, WB_E4M3 = 1 } wb_dtype;

/* The three encoder layer sites of the showcase site's precision table
 * ("The Approach"): encoder_attn_qkv, encoder_attn_out, encoder_ffn (FC1 and
 * FC2).  Weight and activation of one site must have the same type (the
 * tensor core multiplies bf16 by bf16 or E4M3 by E4M3); a mixed site returns
 * WB_EUNSUPPORTED.  Presets: all WB_BF16 ("full" precision, bf16 replacing
 * the pages' fp16), and mixed_fp8 = qkv and ffn E4M3, out bf16. */
typedef struct {
  int32_t qkv_w, qkv_a;
  int32_t out_w, out_a;
  int32_t ffn_w, ffn_a;
} wb_precision;

/* Encoder shape.  large-v3: {128, 1280, 20, 32, 5120}; the tiny test shape
 * {80, 384, 6, 1, 1536}.  Requires d_model = 64 * n_heads, d_model and d_ffn
 * multiples of 64, 8 <= n_mels <= 128 and n_mels a multiple of 8. */
typedef struct {
  int32_t n_mels, d_model, n_heads, n_layers, d_ffn;
} wb_dims;

/* Conv stem weights.  Conv weights are bf16 in TAP-MAJOR layout
 * [3][d_model][c_in] (produce it from the PyTorch layout [c_out][c_in][3]
 * with wb_pack_conv_weight); biases are float32 [d_model]. */
typedef struct {
  const void* conv1_w;   /* bf16 [3][d][n_mels] */
  const float* conv1_b;  /* [d] */
  const void* conv2_w;   /* bf16 [3][d][d] */
  const float* conv2_b;  /* [d] */
} wb_stem_weights;

/* One encoder layer.  Linear weights use the PyTorch/HF layout [out, in].
 * w_qkv is the row concatenation of W_q, W_k, W_v ([3d, d]); b_qkv = [b_q, 0,
 * b_v] (Whisper's key projection has no bias).  A weight stored as E4M3 comes
 * with its float32 dequantisation scale s_* (a DEVICE scalar, as written by
 * wb_quantize_fp8); for bf16 weights s_* is ignored and may be NULL.
 * LayerNorm parameters and biases are float32. */
typedef struct {
  const float* ln1_g;
  const float* ln1_b;
  const void* w_qkv;  const float* b_qkv;  const float* s_qkv;  /* [3d, d], [3d] */
  const void* w_out;  const float* b_out;  const float* s_out;  /* [d, d],  [d]  */
  const float* ln2_g;
  const float* ln2_b;
  const void* w_fc1;  const float* b_fc1;  const float* s_fc1;  /* [F, d],  [F]  */
  const void* w_fc2;  const float* b_fc2;  const float* s_fc2;  /* [d, F],  [d]  */
  /* Optional LayerNorm folds made by wb_fold_layernorm (all three NULL: not folded).  When a bf16
   * QKV (FC1) site has them, the forward skips the LN1 (LN2) pass: the GEMM reads the residual
   * stream itself with w_*_ln and the epilogue applies the row's mean and rstd (see
   * wb_fold_layernorm).  Those statistics come from the residual GEMM that wrote the stream (the
   * out-projection for LN2, the previous layer's FC2 for LN1: per 32-column group, merged per row
   * by a short pass); the first layer of a call forms its LN1 statistics with a pass over x0.
   * E4M3 sites ignore them. */
  const void* w_qkv_ln;  const float* c_qkv;  const float* b_qkv_ln;  /* bf16 [3d, d], f32 [3d], [3d] */
  const void* w_fc1_ln;  const float* c_fc1;  const float* b_fc1_ln;  /* bf16 [F, d],  f32 [F],  [F]  */
} wb_layer_weights;

typedef struct {
  const float* g;
  const float* b;
} wb_ln_weights;

/* ------------------------------------------------------------------------ */

/* Human-readable name of a status code (static string). */
const char* wb_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int wb_version(void);

/* 1 if this library was built with the debug bounds checks (-DWB_DEBUG), else 0.
 * In a debug build every kernel load or store that does not go through a TMA
 * tensor map checks its index against the extent of the buffer it addresses;
 * an index outside is skipped and recorded in the device error word (bit 1,
 * site in bits 8..15).  The arithmetic is otherwise the release build's. */
int wb_debug_build(void);

/* Synchronizes `stream`, then reads and clears this device's error words.
 * Returns WB_ETIMEOUT if any kernel recorded a bounded-wait timeout since the
 * last call, else WB_EBOUNDS if a debug build's bounds check fired, WB_ECUDA
 * if the synchronization itself failed, else WB_OK.  *detail (optional)
 * receives the raw word (bit 0 timeout, bit 1 bounds, bits 8..15 the site). */
wb_status wb_check_device_error(void* stream, uint32_t* detail);

/* Wait site that wb_selftest_wait_timeout() records (bits 8..15 of the word). */
#define WB_SELFTEST_WAIT_SITE 0x7Fu

/* Site that wb_selftest_bounds_check() records (bits 8..15 of the word). */
#define WB_SELFTEST_BOUNDS_SITE 0x7Eu

/* Diagnostic of the debug bounds checks (no memory touched).  Launches one
 * kernel on `stream` that evaluates a bounds check on an index just past the
 * extent it states.  In a debug build (wb_debug_build() == 1) the check fails
 * and records the bounds bit and WB_SELFTEST_BOUNDS_SITE in the device error
 * word, so the next wb_check_device_error() returns WB_EBOUNDS; a release
 * build compiles the check away and records nothing.  Returns WB_ECUDA if the
 * launch fails, else WB_OK (asynchronously). */
wb_status wb_selftest_bounds_check(void* stream);

/* Diagnostic of the bounded-wait path (no compute).  Launches one kernel on
 * `stream` whose single thread waits on an mbarrier that nothing arrives on.
 * The wait gives up after its time limit (about 2 s), sets the timeout bit and
 * WB_SELFTEST_WAIT_SITE in the device error word, and the kernel returns
 * normally: the context stays usable.  The next wb_check_device_error() then
 * returns WB_ETIMEOUT and clears the word.  Returns WB_ECUDA if the launch
 * fails, else WB_OK (asynchronously; nothing else is touched). */
wb_status wb_selftest_wait_timeout(void* stream);

/* --- log-mel front end -----------------------------------------------------
 * The showcase site, "The Solution" (mel_spectrogram.cu card: STFT, mel
 * filterbank, overlapping-chunk mode for long audio) and the PyPI page,
 * "Quick Start" (float32 mono audio at 16 kHz).
 *
 * Chunk c covers samples [c*chunk_stride, c*chunk_stride + 480000) of
 * `audio`, zero-filled past n_samples (chunk_stride = 480000 for a batch of
 * independent 30 s chunks stored back to back; 400000 for 30 s windows at a
 * 25 s stride over one long recording).  Per chunk: reflect pad 200, periodic
 * Hann n_fft 400, hop 160, power spectrum of frames 0..2999 (the last frame
 * is dropped), Slaney mel filterbank over 0-8 kHz, log10(max(., 1e-10)),
 * clamp to (chunk max - 8), then (x + 4) / 4.
 * out: float32 [n_chunks, n_mels, 3000].  n_chunks = 0 is a no-op.
 * Mono only: average multi-channel audio before the call. */
size_t wb_logmel_workspace_bytes(int n_chunks, int n_mels);
wb_status wb_logmel(const float* audio, int64_t n_samples, int64_t chunk_stride, int n_chunks, int n_mels,
                    float* out, void* workspace, size_t workspace_bytes, void* stream);

/* --- log-mel without a workspace -----------------------------------------------
 * The source pages have no counterpart to this entry point.  It is for callers
 * that cannot allocate device memory: a real-time audio thread must not block
 * in cudaMalloc (which can synchronize the device), and plugin hosts or
 * serving runtimes that own every device buffer forbid their plugins to
 * allocate.  It computes exactly what wb_logmel computes, but takes its
 * scratch from one fixed array built into the library (about 13 MiB, present
 * on every device that loads the library until the process exits) instead of
 * a caller workspace.  It calls no allocating routine.
 *  - n_chunks above WB_LOGMEL_STATIC_MAX_CHUNKS returns WB_EINVAL before
 *    anything is launched; other arguments as for wb_logmel.
 *  - The first call on a device, made with that device current, looks up the
 *    array's device address; make that first call before any stream capture.
 *    The address is kept for the life of the process: after cudaDeviceReset()
 *    of that device it is stale, so do not call this entry point on a device
 *    that was reset in the same process.
 *  - All calls share the one array per device and it keeps the previous
 *    call's contents (the call clears what must start at zero itself).  Calls
 *    whose GPU work overlaps, e.g. on two streams without ordering, race on
 *    it: issue them on one stream or order them. */
#define WB_LOGMEL_STATIC_MAX_CHUNKS 2
wb_status wb_logmel_static(const float* audio, int64_t n_samples, int64_t chunk_stride, int n_chunks, int n_mels,
                           float* out, void* stream);

/* --- conv stem ---------------------------------------------------------------
 * x0[b] = GELU(conv2(GELU(conv1(logmel[b])))) + sinusoidal positions, with
 * conv1 = Conv1d(n_mels -> d, k3, stride 1, pad 1) and conv2 = Conv1d(d -> d,
 * k3, stride 2, pad 1), computed as implicit GEMMs on the tensor cores
 * (bf16 operands, fp32 accumulation, exact-erf GELU).
 * logmel: float32 [batch, n_mels, 3000]; x0: bf16 [batch, 1500, d]. */
size_t wb_conv_stem_workspace_bytes(const wb_dims* dims, int batch);
wb_status wb_conv_stem(const float* logmel, int batch, const wb_dims* dims, const wb_stem_weights* w, void* x0,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Reorders a PyTorch Conv1d weight (float32 [c_out][c_in][3]) into the
 * tap-major bf16 layout [3][c_out][c_in] that wb_stem_weights expects. */
wb_status wb_pack_conv_weight(const float* w, int c_out, int c_in, void* packed, void* stream);

/* --- encoder -----------------------------------------------------------------
 * Runs pre-LN encoder layers [layer_begin, layer_end) of `layers` on x0
 * (bf16 [batch, 1500, d]) and, if apply_final_ln, the final LayerNorm
 * (ln_post); writes bf16 [batch, 1500, d] to `out` (which must not alias x0).
 * Per layer: h += OutProj(Attn(QKV(LN1(h)))); h += FC2(GELU(FC1(LN2(h)))),
 * LayerNorm eps 1e-5 (PyPI page, "Direct Kernel API"), softmax attention over
 * all 1500 positions with scale 1/8, erf GELU.  `precision` selects the
 * operand type of each site.  An E4M3 activation is quantised on the device
 * with an absmax scale per tensor (showcase site, "Learnings": scales from
 * activation maxima), the tensor being one 30 s chunk's [1500, k] operand:
 * every chunk gets its own scale, so a chunk's result does not depend on the
 * other chunks of the batch.  layers[i] is read only for begin <= i < end. */
size_t wb_encoder_workspace_bytes(const wb_dims* dims, int batch, const wb_precision* precision);
wb_status wb_encoder_forward(const void* x0, int batch, const wb_dims* dims, const wb_layer_weights* layers,
                             const wb_ln_weights* ln_post, const wb_precision* precision, int layer_begin,
                             int layer_end, int apply_final_ln, void* out, void* workspace, size_t workspace_bytes,
                             void* stream);

/* --- end to end from host memory -------------------------------------------------
 * The PyPI page, "Quick Start" and "Batch Transcription": the caller hands over float32
 * 16 kHz audio held in HOST memory and receives the encoder's hidden states in HOST memory.
 * wb_encode_host runs n_batches batches through wb_logmel, wb_conv_stem and
 * wb_encoder_forward (layers 0 .. dims.n_layers - 1 and the final LayerNorm): for batch i,
 * one cudaMemcpyAsync of host_audio[i] (samples_per_batch floats) into a device audio
 * buffer, the three calls on `stream`, and one cudaMemcpyAsync of the bf16
 * [batch, 1500, d] result into host_out[i].
 *  - With upload_stream and download_stream set (both or neither), uploads and downloads
 *    run on them, against two device audio and two device output buffers, so that the
 *    copies of neighbouring batches overlap a batch's compute; CUDA events order each
 *    buffer's reuse (the call creates and destroys 10 events; it allocates no memory).
 *    With both NULL every copy runs in order on `stream` and only dev_audio[0] and
 *    dev_out[0] are used.
 *  - Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister): copies from
 *    pageable memory are correct but do not overlap.
 *  - Returns once everything is queued; all of it, the last download included, is ordered
 *    before later work on `stream` (synchronize `stream` to wait for host_out).
 *  - Every pointer in the struct is a DEVICE pointer owned by the caller, except the
 *    weight structs (host structs holding device pointers) and the streams.  Workspaces as
 *    the *_workspace_bytes() queries give for (dims, batch, precision).
 *  - WB_EINVAL for a missing buffer or host pointer, n_batches < 0, or only one copy
 *    stream; otherwise the status of the first call that fails (nothing after it is
 *    queued; earlier batches may already be in flight). */
typedef struct {
  wb_dims dims;
  int32_t batch;                  /* chunks per batch */
  int64_t samples_per_batch;      /* floats per host_audio[i] (wb_logmel's n_samples) */
  int64_t chunk_stride;           /* as for wb_logmel: 480000, or 400000 for 25 s strides */
  const wb_stem_weights* stem;
  const wb_layer_weights* layers; /* [dims.n_layers] */
  const wb_ln_weights* ln_post;
  wb_precision precision;
  float* dev_audio[2];            /* f32 [samples_per_batch] each */
  float* dev_mel;                 /* f32 [batch, n_mels, 3000] */
  void* dev_x0;                   /* bf16 [batch, 1500, d] */
  void* dev_out[2];               /* bf16 [batch, 1500, d] each */
  void* ws_mel;                   /* wb_logmel_workspace_bytes(batch, n_mels) */
  size_t ws_mel_bytes;
  void* ws_stem;                  /* wb_conv_stem_workspace_bytes(&dims, batch) */
  size_t ws_stem_bytes;
  void* ws_enc;                   /* wb_encoder_workspace_bytes(&dims, batch, &precision) */
  size_t ws_enc_bytes;
  void* upload_stream;            /* cudaStream_t for host -> device copies, or NULL */
  void* download_stream;          /* cudaStream_t for device -> host copies, or NULL */
} wb_host_pipeline;
wb_status wb_encode_host(const wb_host_pipeline* p, const float* const* host_audio, void* const* host_out,
                         int n_batches, void* stream);

/* --- FP8 E4M3 ------------------------------------------------------------------
 * PyPI page, "Direct Kernel API" (quantise_e4m3 / dequantise_e4m3) and the
 * showcase site, "The Solution" (fp8_quantize.cu: per-tensor scale, amax).
 * quantize: amax = max|x| over the n bf16 values, inv = 448 / amax, code =
 * E4M3(x * inv) rounded to nearest even and saturated to +-448; *scale (a
 * DEVICE float) receives amax / 448 (1 when amax = 0).  dequantize: y =
 * decode(q) * (*scale) as bf16. */
wb_status wb_quantize_fp8(const void* x, int64_t n, uint8_t* q, float* scale, void* stream);
wb_status wb_dequantize_fp8(const uint8_t* q, const float* scale, int64_t n, void* y, void* stream);

/* --- LayerNorm folded into the linear layer after it ---------------------------
 * The pre-LN layer computes y = LN(x; gamma, beta) W^T + b with LN(x) = (x - mean) rstd gamma + beta
 * (PyPI page, "Direct Kernel API": eps 1e-5).  By that definition
 *   y[n] = rstd (x . w_ln[n] - mean c[n]) + b_ln[n],  w_ln = W diag(gamma),
 *   c[n] = sum_k w_ln[n,k],  b_ln[n] = b[n] + sum_k beta[k] W[n,k],
 * so a GEMM can read x itself and apply the row statistics in its epilogue.  (The pages have no
 * counterpart: this is a rewrite of the LayerNorm definition, not a step they describe.)
 * Writes w_ln = bf16(W[n,k] gamma[k]) (bf16 [n_out, d]) and, in float32, c (from the rounded w_ln)
 * and b_ln ([n_out] each).  w: bf16 [n_out, d]; b may be NULL (zero); gamma, beta: float32 [d].
 * All pointers are device pointers owned by the caller, 16-byte aligned; d % 8 == 0.
 * WB_EINVAL for a missing pointer, bad alignment or size. */
wb_status wb_fold_layernorm(const void* w, const float* b, const float* gamma, const float* beta, int n_out, int d,
                            void* w_ln, float* c, float* b_ln, void* stream);

/* --- building blocks (exposed for unit tests and custom pipelines) ------------
 * wb_linear: out[m, n] = act(alpha * sum_k a[m, k] w[n, k] + bias[n]) + resid[m, n]
 * with alpha = (*scale_a) * (*scale_w) for E4M3 operands (both must then be
 * given) and 1 for bf16; act = exact-erf GELU when gelu != 0.  a: [M, K],
 * w: [N, K] (bf16 or E4M3 per `dtype`), bias float32 [N] or NULL, resid bf16
 * [M, N] or NULL, out bf16 [M, N].  N must be a multiple of 32 and K a
 * multiple of 8 (bf16) or 16 (E4M3). */
wb_status wb_linear(const void* a, const void* w, int M, int N, int K, int dtype, const float* bias,
                    const float* scale_a, const float* scale_w, int gelu, const void* resid, void* out,
                    void* stream);

/* Fused residual + LayerNorm (PyPI page, "Direct Kernel API":
 * layernorm_fused / layernorm_fused_residual): total = x + residual,
 * y = (total - mean) / sqrt(var + eps) * g + b over rows of width d (biased
 * variance).  residual and total may be NULL.  x, residual, total, y: bf16
 * [rows, d]; g, b: float32 [d], 16-byte aligned.  d must be a multiple of 128 and <= 2048. */
wb_status wb_layernorm(const void* x, const void* residual, const float* g, const float* b, int rows, int d,
                       float eps, void* y, void* total, void* stream);

/* Softmax attention without a mask (the encoder's self-attention):
 * out[b, t, h*64:(h+1)*64] = softmax(q_h k_h^T / 8) v_h for every batch item
 * and head.  q, k, v, out: bf16 [batch, T, 64*n_heads].  Needs a workspace of
 * wb_attention_workspace_bytes() for the transposed V. */
size_t wb_attention_workspace_bytes(int batch, int T, int n_heads);
wb_status wb_attention(const void* q, const void* k, const void* v, int batch, int T, int n_heads, void* out,
                       void* workspace, size_t workspace_bytes, void* stream);

/* LayerNorm straight to FP8 E4M3 codes with one absmax scale per batch item
 * (the pages' per-tensor-scaled E4M3 activations, one tensor per 30 s chunk):
 * y = LN(x) as wb_layernorm computes it, rounded to bf16; amax[i] = max |y|
 * over the rows of item i (rows i*rows_per_item .. (i+1)*rows_per_item - 1);
 * q = E4M3_rn_satfinite(y * 448 / amax[i]) (scale 1 where amax[i] == 0), so
 * y ~ q * amax[i] / 448.  The arithmetic of wb_layernorm followed by
 * wb_quantize_fp8 of each item, without the bf16 round trip through memory
 * (two passes over x: statistics + absmax, then codes); the row statistics
 * are summed in another order, so a value lying on a rounding boundary can
 * come out one bf16 / E4M3 step away from that two-call result.
 * x: bf16 [rows, d]; g, b: float32 [d]; q: u8 [rows, d]; amax: float32
 * [ceil(rows / rows_per_item)], overwritten; stats: float32 [rows][2] out,
 * each row's (mean, rstd).  16-byte aligned (amax 4-byte); d a multiple of
 * 128, <= 2048.  WB_EINVAL for bad sizes, pointers or alignment. */
wb_status wb_layernorm_e4m3(const void* x, const float* g, const float* b, int rows, int d, float eps,
                            int rows_per_item, uint8_t* q, float* amax, float* stats, void* stream);

/* --- after the encoder: decoder cross-attention keys and values ---------------------
 * The showcase site, "The Solution" (decoder cross-attention is one of the three
 * attention patterns) and "The Approach" (decoder_cross_attn site): every decoder
 * layer projects the encoder output to its own keys and values once per audio
 * chunk.  For decoder layer l: K_l = enc_out Wk_l^T, V_l = enc_out Wv_l^T + bv_l
 * (Whisper's key projection has no bias).  w[l].w_kv is bf16 [2d, d] = [Wk_l; Wv_l]
 * (HF layout), w[l].b_kv float32 [2d] = [0, bv_l].  enc_out: bf16 [batch, 1500, d];
 * kv: bf16 [n_dec_layers][batch * 1500][2d] with K in columns 0..d-1 and V in d..2d-1. */
typedef struct {
  const void* w_kv;
  const float* b_kv;
} wb_cross_kv_weights;
wb_status wb_cross_kv(const void* enc_out, int batch, const wb_dims* dims, int n_dec_layers,
                      const wb_cross_kv_weights* w, void* kv, void* stream);

/* Fused residual + RMSNorm (PyPI page, "Direct Kernel API": rmsnorm_fused):
 * total = x + residual, y = total / sqrt(mean(total^2) + eps) * g.  As wb_layernorm
 * without beta; residual and total may be NULL. */
wb_status wb_rmsnorm(const void* x, const void* residual, const float* g, int rows, int d, float eps, void* y,
                     void* total, void* stream);

/* FP8 E5M2 casts with one per-tensor scale (showcase site, "The Solution": casts for both
 * E4M3 and E5M2, E5M2 for more range): amax = max|x|, code = E5M2(x * 57344 / amax)
 * rounded to nearest even and saturated to +-57344; *scale (device) = amax / 57344
 * (1 when amax = 0). */
wb_status wb_quantize_e5m2(const void* x, int64_t n, uint8_t* q, float* scale, void* stream);
wb_status wb_dequantize_e5m2(const uint8_t* q, const float* scale, int64_t n, void* y, void* stream);

/* --- kernel timing (benchmarks) -------------------------------------------------
 * Between wb_profile_begin() and wb_profile_end() every kernel that libwb
 * launches is bracketed by two CUDA events recorded on its launch stream.
 * wb_profile_end() waits for those events, fills up to max_classes entries
 * (static class names such as "enc.fc1", summed device milliseconds, and the
 * number of kernels launched in that class), disables timing and returns the
 * number of classes.  Any array may be NULL.  Host-side bookkeeping only: use
 * it from one thread, on one device at a time. */
wb_status wb_profile_begin(void);
int wb_profile_end(int max_classes, const char** names, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif
#endif /* WB_H */
