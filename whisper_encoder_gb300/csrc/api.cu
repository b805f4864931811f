// libwb C ABI: argument checks, workspace layout, TMA tensor maps and the
// launch sequence of each entry point declared in include/wb.h.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/wb.h"
#include "internal.h"

using namespace wb;

namespace {

// ------------------------------ device error word --------------------------
__device__ uint32_t g_err_word;

constexpr int MAX_DEVICES = 64;
uint32_t* g_err_ptr[MAX_DEVICES] = {nullptr};
std::mutex g_mu;

uint32_t* err_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[dev];
}

// ------------------------------ tensor maps --------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool encoder_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// rank-dimensional tiled map; strides in bytes for dims 1..rank-1; 128-byte swizzle.
bool make_map(CUtensorMap* m, bool u8, int rank, const void* base, const uint64_t* dims, const uint64_t* strides,
              const uint32_t* box, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B, bool f16 = false) {
  if (!encoder_fn()) return false;
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  CUresult r = g_encode(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A operand view: (k, row, part, batch) with box (BK, 128, 1, 1).
bool a_map(CUtensorMap* m, bool u8, const void* base, uint64_t k, uint64_t rows, uint64_t parts, uint64_t batch,
           uint64_t row_stride, uint64_t part_stride, uint64_t batch_stride) {
  const uint64_t dims[4] = {k, rows, parts, batch};
  const uint64_t str[3] = {row_stride, part_stride, batch_stride};
  const uint32_t box[4] = {u8 ? 128u : 64u, static_cast<uint32_t>(GEMM_BM), 1u, 1u};
  return make_map(m, u8, 4, base, dims, str, box);
}

// B operand view: (k, n, part) with box (BK, BN, 1).
bool b_map(CUtensorMap* m, bool u8, const void* base, uint64_t k, uint64_t n, uint64_t parts, uint64_t row_stride,
           uint64_t part_stride, int bn) {
  const uint64_t dims[3] = {k, n, parts};
  const uint64_t str[2] = {row_stride, part_stride};
  const uint32_t box[3] = {u8 ? 128u : 64u, static_cast<uint32_t>(bn), 1u};
  return make_map(m, u8, 3, base, dims, str, box);
}


// Output / residual view for the standard epilogues: (n, row, item) with 32 x 32 boxes and the
// 64-byte swizzle the epilogue writes its staging boxes in.
bool o_map(CUtensorMap* m, const void* base, uint64_t n, uint64_t rows, uint64_t items, uint64_t ld_elems,
           uint64_t item_elems) {
  const uint64_t dims[3] = {n, rows, items};
  const uint64_t str[2] = {ld_elems * 2, item_elems * 2};
  const uint32_t box[3] = {32u, 32u, 1u};
  return make_map(m, false, 3, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// ------------------------------ kernel timing -------------------------------
// While enabled, every libwb launch is bracketed by two CUDA events recorded
// on its own stream; wb_profile_end() sums the elapsed times per kernel class.
enum ProfClass {
  PC_LOGMEL_PREP, PC_LOGMEL_DFT, PC_LOGMEL_MEL, PC_LOGMEL_POST, PC_STEM_PREP, PC_STEM_CONV1, PC_STEM_CONV2,
  PC_ENC_LN, PC_ENC_QUANT, PC_ENC_QKV, PC_ENC_ATTN, PC_ENC_OUT, PC_ENC_FC1, PC_ENC_FC2, PC_OTHER, PC_COUNT
};
const char* const kProfNames[PC_COUNT] = {
    "logmel.prep", "logmel.dft", "logmel.mel", "logmel.post", "stem.prep", "stem.conv1", "stem.conv2",
    "enc.layernorm", "enc.quantize", "enc.qkv", "enc.attention", "enc.out_proj", "enc.fc1", "enc.fc2", "other"};

struct ProfRec {
  int cls, kernels;
  cudaEvent_t a, b;
};
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

struct Prof {
  int cls, kernels;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  Prof(int c, cudaStream_t st, int k = 1) : cls(c), kernels(k), s(st) {
    if (!g_prof_on) return;
    std::lock_guard<std::mutex> lk(g_mu);
    a = prof_event();
    if (a) cudaEventRecord(a, s);
  }
  ~Prof() {
    if (!a) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t b = prof_event();
    if (!b) return;
    cudaEventRecord(b, s);
    g_prof_recs.push_back(ProfRec{cls, kernels, a, b});
  }
};

// ------------------------------ helpers ------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return o;
  }
};

#define WB_CUDA(x)                         \
  do {                                     \
    if ((x) != cudaSuccess) return WB_ECUDA; \
  } while (0)

GemmParams base_params() {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.batch = 1;
  p.rows_per_item = T_TOK;
  p.err = err_ptr();
  return p;
}

void one_pass(GemmParams& p, int n_kb) {
  p.n_pass = 1;
  p.pass[0] = GemmPass{0, 0, 0, 0, 0, 0, static_cast<int16_t>(n_kb), 0};
}

// Plain GEMM out[M, N] = epilogue(A[M, K] . W[N, K]^T), A and W dense row-major; the output
// (and residual) rows are ldo elements apart, and the output map covers its first n_store columns.
// Tile width for an M x N output (per batch item, `items` items).  Wide N takes 256-column tiles; when M
// is small (a few chunks) 128-wide tiles are used if the waves they need, at about 0.7 of a 256-wide
// tile's time each (half the work, a less efficient MMA shape; measured 0.65-0.74 at N = 1280), finish
// sooner than the 256-wide waves.
int pick_bn(long long M, long long items, int N) {
  if (!(N % 256 == 0 || N > 512)) return 128;
  const long long sms = sm_count(), mt = items * ((M + GEMM_BM - 1) / GEMM_BM);
  const long long w256 = (mt * ((N + 255) / 256) + sms - 1) / sms;
  const long long w128 = (mt * ((N + 127) / 128) + sms - 1) / sms;
  return 7 * w128 < 10 * w256 ? 128 : 256;
}

wb_status dense_gemm(const void* A, const void* W, int M, int N, int K, bool fp8, int epi, void* out, long long ldo,
                     int n_store, const void* resid, GemmParams p, cudaStream_t s, int prof_cls = PC_OTHER) {
  GemmLaunch g;
  std::memset(&g, 0, sizeof(g));
  const uint64_t es = fp8 ? 1 : 2;
  g.bn = pick_bn(M, 1, N);
  g.fp8 = fp8;
  g.epi = epi;
  if (!a_map(&g.amap[0], fp8, A, K, M, 1, 1, K * es, static_cast<uint64_t>(M) * K * es,
             static_cast<uint64_t>(M) * K * es))
    return WB_ECUDA;
  g.amap[1] = g.amap[2] = g.amap[3] = g.amap[0];
  if (!b_map(&g.bmap, fp8, W, K, N, 1, K * es, static_cast<uint64_t>(N) * K * es, g.bn)) return WB_ECUDA;
  if (!o_map(&g.omap, out, n_store, M, 1, ldo, static_cast<uint64_t>(M) * ldo)) return WB_ECUDA;
  p.resid = static_cast<const __nv_bfloat16*>(resid);
  p.resid_ld = ldo;
  p.resid_item = static_cast<long long>(M) * ldo;
  p.resid_elems = static_cast<long long>(M) * ldo;
  p.amax_items = p.rows_per_item > 0 ? (M + p.rows_per_item - 1) / p.rows_per_item : 0;
  p.M = M;
  p.N = N;
  p.batch = 1;
  const int bk = fp8 ? 128 : 64;
  one_pass(p, (K + bk - 1) / bk);
  g.p = p;
  {
    Prof pr(prof_cls, s);
    WB_CUDA(launch_gemm(g, s));
  }
  return WB_OK;
}

bool dims_ok(const wb_dims* d) {
  return d && d->n_heads > 0 && d->d_model == 64 * d->n_heads && d->d_model % 64 == 0 && d->d_ffn > 0 &&
         d->d_ffn % 64 == 0 && d->n_mels >= 8 && d->n_mels <= MEL_ROWS && d->n_mels % 8 == 0 && d->n_layers >= 0 &&
         d->d_model <= 2048;
}

bool site_ok(int w, int a) { return (w == WB_BF16 || w == WB_E4M3) && w == a; }

struct EncLayout {
  size_t h, a, qk, vt, o, g, aq, gq, slots, stats, ln_part, total;
};

EncLayout enc_layout(const wb_dims* d, int batch, const wb_precision* pr) {
  const size_t M = static_cast<size_t>(batch) * T_TOK;
  const size_t D = d->d_model, F = d->d_ffn;
  const bool any8 = pr && (pr->qkv_a == WB_E4M3 || pr->out_a == WB_E4M3 || pr->ffn_a == WB_E4M3);
  const bool ffn8 = pr && pr->ffn_a == WB_E4M3;
  Carver c;
  EncLayout L;
  L.h = c.take(M * D * 2);
  L.a = c.take(M * D * 2);
  L.qk = c.take(M * 2 * D * 2);
  L.vt = c.take(static_cast<size_t>(batch) * d->n_heads * 64 * T_PAD * 2);
  L.o = c.take(M * D * 2);
  L.g = c.take(M * F * 2);
  L.aq = any8 ? c.take(M * D) : 0;
  L.gq = ffn8 ? c.take(M * F) : 0;
  // per layer, per E4M3 operand site (qkv, out, fc1, fc2 inputs), per batch item: one absmax
  L.slots = c.take(static_cast<size_t>(4) * (d->n_layers > 0 ? d->n_layers : 1) * batch * sizeof(float));
  // LayerNorm row statistics (mean, rstd) for a folded LN1 / LN2 site
  L.stats = c.take(M * sizeof(float2));
  // (mean, M2) per row and 32-column group, left by the residual GEMMs' epilogues
  L.ln_part = c.take(M * (D / 32) * sizeof(float2));
  L.total = c.off;
  return L;
}

struct MelLayout {
  size_t xs, basis, pw, fbs, mmax, total;
};

MelLayout mel_layout(int n_chunks) {
  Carver c;
  MelLayout L;
  L.xs = c.take(static_cast<size_t>(n_chunks) * 3 * PADDED * 2);
  L.basis = c.take(static_cast<size_t>(3) * DFT_ROWS * N_FFT * 2);
  L.pw = c.take(static_cast<size_t>(n_chunks) * 2 * N_FRAMES * N_BIN_PAD * 2);
  L.fbs = c.take(static_cast<size_t>(2) * MEL_ROWS * N_BIN_PAD * 2);
  L.mmax = c.take(static_cast<size_t>(n_chunks) * sizeof(float));
  L.total = c.off;
  return L;
}

struct StemLayout {
  size_t yTp, y1p, pos, total;
};

StemLayout stem_layout(const wb_dims* d, int batch) {
  Carver c;
  StemLayout L;
  L.yTp = c.take(static_cast<size_t>(batch) * (N_FRAMES + 2) * d->n_mels * 2);
  L.y1p = c.take(static_cast<size_t>(batch) * (N_FRAMES + 1) * d->d_model * 2);
  L.pos = c.take(static_cast<size_t>(T_TOK) * d->d_model * sizeof(float));   // position table
  L.total = c.off;
  return L;
}

// Attention over q/k row views (row stride ld_qk elements) and V^T.
wb_status run_attention(const __nv_bfloat16* q, const __nv_bfloat16* k, long long ld_qk, const __half* vt,
                        int batch, int T, int H, __nv_bfloat16* out, cudaStream_t s, float* amax = nullptr) {
  const uint64_t d = static_cast<uint64_t>(H) * 64;
  CUtensorMap qm, km, vm;
  const uint64_t qdims[3] = {d, static_cast<uint64_t>(T), static_cast<uint64_t>(batch)};
  const uint64_t qstr[2] = {static_cast<uint64_t>(ld_qk) * 2, static_cast<uint64_t>(ld_qk) * 2 * T};
  const uint32_t qbox[3] = {64, ATT_BQ, 1};
  const uint32_t kbox[3] = {64, ATT_BKV, 1};
  if (!make_map(&qm, false, 3, q, qdims, qstr, qbox)) return WB_ECUDA;
  if (!make_map(&km, false, 3, k, qdims, qstr, kbox)) return WB_ECUDA;
  const uint64_t vdims[3] = {static_cast<uint64_t>(T), 64, static_cast<uint64_t>(batch) * H};
  const uint64_t vstr[2] = {static_cast<uint64_t>(T_PAD) * 2, static_cast<uint64_t>(T_PAD) * 2 * 64};
  const uint32_t vbox[3] = {64, 64, 1};
  if (!make_map(&vm, false, 3, vt, vdims, vstr, vbox, CU_TENSOR_MAP_SWIZZLE_128B, true)) return WB_ECUDA;
  AttnParams p;
  p.T = T;
  p.H = H;
  p.d = static_cast<int>(d);
  p.batch = batch;
  p.scale_log2 = 1.4426950408889634f / 8.0f;
  p.out = out;
  p.amax = amax;
  p.err = err_ptr();
  Prof pr(PC_ENC_ATTN, s);
  WB_CUDA(launch_attention(qm, km, vm, p, s));
  return WB_OK;
}

}  // namespace

// ============================================================================
extern "C" {

const char* wb_status_string(int status) {
  switch (status) {
    case WB_OK: return "ok";
    case WB_EINVAL: return "invalid argument";
    case WB_ECUDA: return "CUDA error";
    case WB_EUNSUPPORTED: return "unsupported configuration";
    case WB_ETIMEOUT: return "device-side wait timed out";
    case WB_EWORKSPACE: return "workspace missing or too small";
    case WB_EBOUNDS: return "a debug build's bounds check found an index outside its buffer";
    default: return "unknown status";
  }
}

int wb_version(void) { return 100; }

int wb_debug_build(void) {
#ifdef WB_DEBUG
  return 1;
#else
  return 0;
#endif
}

wb_status wb_check_device_error(void* stream, uint32_t* detail) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return WB_ECUDA;
  // the tensor-core kernels' word and the SIMT kernels' word (bounds checks of debug builds)
  uint32_t* words[2] = {err_ptr(), simt_err_ptr()};
  uint32_t word = 0;
  for (uint32_t* e : words) {
    if (!e) return WB_ECUDA;
    uint32_t w = 0;
    if (cudaMemcpy(&w, e, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return WB_ECUDA;
    if (w) {
      const uint32_t zero = 0;
      if (cudaMemcpy(e, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return WB_ECUDA;
    }
    word |= w;
  }
  if (detail) *detail = word;
  if (word & ERR_TIMEOUT) return WB_ETIMEOUT;
  return (word & ERR_BOUNDS) ? WB_EBOUNDS : WB_OK;
}

wb_status wb_selftest_bounds_check(void* stream) {
  if (!simt_err_ptr()) return WB_ECUDA;
  WB_CUDA(launch_bounds_check_selftest(WB_SELFTEST_BOUNDS_SITE, static_cast<cudaStream_t>(stream)));
  return WB_OK;
}

wb_status wb_selftest_wait_timeout(void* stream) {
  uint32_t* e = err_ptr();
  if (!e) return WB_ECUDA;
  WB_CUDA(launch_wait_timeout_selftest(e, WB_SELFTEST_WAIT_SITE, static_cast<cudaStream_t>(stream)));
  return WB_OK;
}

// ------------------------------- log-mel -----------------------------------
size_t wb_logmel_workspace_bytes(int n_chunks, int n_mels) {
  (void)n_mels;
  return n_chunks > 0 ? mel_layout(n_chunks).total : 0;
}

wb_status wb_logmel(const float* audio, int64_t n_samples, int64_t chunk_stride, int n_chunks, int n_mels,
                    float* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_chunks < 0 || n_mels < 8 || n_mels > MEL_ROWS || n_mels % 8 != 0 || n_samples < 0 || chunk_stride < 1)
    return WB_EINVAL;
  if (n_chunks == 0) return WB_OK;
  if (!audio || !out || !aligned16(out) || !aligned16(audio)) return WB_EINVAL;
  const MelLayout L = mel_layout(n_chunks);
  if (!workspace || !aligned16(workspace) || workspace_bytes < L.total) return WB_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto* xs = reinterpret_cast<__nv_bfloat16*>(ws + L.xs);
  auto* basis = reinterpret_cast<__nv_bfloat16*>(ws + L.basis);
  auto* pw = reinterpret_cast<__nv_bfloat16*>(ws + L.pw);
  auto* fbs = reinterpret_cast<__nv_bfloat16*>(ws + L.fbs);
  auto* mmax = reinterpret_cast<float*>(ws + L.mmax);

  WB_CUDA(cudaMemsetAsync(mmax, 0, n_chunks * sizeof(float), s));
  {
    Prof pr(PC_LOGMEL_PREP, s, 3);
    WB_CUDA(launch_dft_basis(basis, s));
    WB_CUDA(launch_mel_fb(fbs, n_mels, s));
    WB_CUDA(launch_pad_split(audio, n_samples, chunk_stride, n_chunks, xs, s));
  }

  // Windowed DFT: frames are read as four column segments of the padded
  // signal (row t starts at sample 160 t), each times its slice of the basis,
  // for the six leading products of the 3-way bf16 split.
  {
    GemmLaunch g;
    std::memset(&g, 0, sizeof(g));
    g.bn = 256;
    g.fp8 = false;
    g.epi = EPI_POWER;
    for (int sgm = 0; sgm < 4; ++sgm) {
      if (!a_map(&g.amap[sgm], false, xs + 128 * sgm, sgm < 3 ? 128 : 64, N_FRAMES, 3, n_chunks, HOP * 2,
                 static_cast<uint64_t>(PADDED) * 2, static_cast<uint64_t>(PADDED) * 2 * 3))
        return WB_ECUDA;
    }
    if (!b_map(&g.bmap, false, basis, N_FFT, DFT_ROWS, 3, N_FFT * 2, static_cast<uint64_t>(DFT_ROWS) * N_FFT * 2, 256))
      return WB_ECUDA;
    GemmParams p = base_params();
    p.M = N_FRAMES;
    p.N = DFT_ROWS;
    p.batch = n_chunks;
    const int pairs[6][2] = {{0, 0}, {0, 1}, {1, 0}, {0, 2}, {1, 1}, {2, 0}};
    int np = 0;
    for (int q = 0; q < 6; ++q)
      for (int sgm = 0; sgm < 4; ++sgm)
        p.pass[np++] = GemmPass{static_cast<int8_t>(sgm), static_cast<int8_t>(pairs[q][0]), 0,
                                static_cast<int8_t>(pairs[q][1]), 0, static_cast<int16_t>(128 * sgm),
                                static_cast<int16_t>(sgm < 3 ? 2 : 1), 0};
    p.n_pass = np;
    p.pw = pw;
    p.pw_ld = N_BIN_PAD;
    p.pw_elems = static_cast<long long>(n_chunks) * 2 * N_FRAMES * N_BIN_PAD;
    g.p = p;
    Prof pr(PC_LOGMEL_DFT, s);
    WB_CUDA(launch_gemm(g, s));
  }
  // Mel filterbank: power (hi, lo) x filterbank (hi, lo), three leading products.
  {
    GemmLaunch g;
    std::memset(&g, 0, sizeof(g));
    g.bn = 128;
    g.fp8 = false;
    g.epi = EPI_MEL;
    if (!a_map(&g.amap[0], false, pw, N_BIN_PAD, N_FRAMES, 2, n_chunks, N_BIN_PAD * 2,
               static_cast<uint64_t>(N_FRAMES) * N_BIN_PAD * 2, static_cast<uint64_t>(N_FRAMES) * N_BIN_PAD * 4))
      return WB_ECUDA;
    g.amap[1] = g.amap[2] = g.amap[3] = g.amap[0];
    if (!b_map(&g.bmap, false, fbs, N_BIN_PAD, MEL_ROWS, 2, N_BIN_PAD * 2,
               static_cast<uint64_t>(MEL_ROWS) * N_BIN_PAD * 2, 128))
      return WB_ECUDA;
    GemmParams p = base_params();
    p.M = N_FRAMES;
    p.N = MEL_ROWS;
    p.batch = n_chunks;
    const int pairs[3][2] = {{0, 0}, {0, 1}, {1, 0}};
    for (int q = 0; q < 3; ++q)
      p.pass[q] = GemmPass{0, static_cast<int8_t>(pairs[q][0]), 0, static_cast<int8_t>(pairs[q][1]), 0, 0,
                           N_BIN_PAD / 64, 0};
    p.n_pass = 3;
    p.mel_out = out;
    p.mel_max = mmax;
    p.n_valid = n_mels;
    p.mel_elems = static_cast<long long>(n_chunks) * n_mels * N_FRAMES;
    g.p = p;
    Prof pr(PC_LOGMEL_MEL, s);
    WB_CUDA(launch_gemm(g, s));
  }
  {
    Prof pr(PC_LOGMEL_POST, s);
    WB_CUDA(launch_logmel_post(out, mmax, n_chunks, n_mels, s));
  }
  return WB_OK;
}

// ------------------------------- conv stem ---------------------------------
size_t wb_conv_stem_workspace_bytes(const wb_dims* dims, int batch) {
  if (!dims_ok(dims) || batch < 1) return 0;
  return stem_layout(dims, batch).total;
}

wb_status wb_pack_conv_weight(const float* w, int c_out, int c_in, void* packed, void* stream) {
  if (!w || !packed || c_out < 1 || c_in < 1) return WB_EINVAL;
  WB_CUDA(launch_pack_conv(w, c_out, c_in, static_cast<__nv_bfloat16*>(packed), static_cast<cudaStream_t>(stream)));
  return WB_OK;
}

wb_status wb_conv_stem(const float* logmel, int batch, const wb_dims* dims, const wb_stem_weights* w, void* x0,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!dims_ok(dims) || batch < 0) return WB_EINVAL;
  if (batch == 0) return WB_OK;
  if (!logmel || !w || !w->conv1_w || !w->conv1_b || !w->conv2_w || !w->conv2_b || !x0 || !aligned16(x0) ||
      !aligned16(w->conv1_w) || !aligned16(w->conv2_w))
    return WB_EINVAL;
  const StemLayout L = stem_layout(dims, batch);
  if (!workspace || !aligned16(workspace) || workspace_bytes < L.total) return WB_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto* yTp = reinterpret_cast<__nv_bfloat16*>(ws + L.yTp);
  auto* y1p = reinterpret_cast<__nv_bfloat16*>(ws + L.y1p);
  auto* pos = reinterpret_cast<float*>(ws + L.pos);
  const int C = dims->n_mels, D = dims->d_model;

  {
    Prof pr(PC_STEM_PREP, s, 5);
    WB_CUDA(launch_stem_transpose(logmel, batch, C, yTp, s));
    WB_CUDA(launch_pos_table(pos, T_TOK, D, s));
    WB_CUDA(launch_zero_rows(y1p, D, static_cast<long long>(N_FRAMES + 1) * D, batch, 0, s));
  }
  {  // conv1: three taps = three passes over row-shifted views of yTp
    GemmLaunch g;
    std::memset(&g, 0, sizeof(g));
    const int bn = D % 256 == 0 ? pick_bn(N_FRAMES, batch, D) : 128;
    g.bn = bn;
    g.epi = EPI_BIAS_GELU;
    const uint64_t rs = static_cast<uint64_t>(C) * 2, item = static_cast<uint64_t>(N_FRAMES + 2) * C * 2;
    if (!a_map(&g.amap[0], false, yTp, C, N_FRAMES + 2, 1, batch, rs, item, item)) return WB_ECUDA;
    g.amap[1] = g.amap[2] = g.amap[3] = g.amap[0];
    if (!b_map(&g.bmap, false, w->conv1_w, C, D, 3, rs, static_cast<uint64_t>(D) * C * 2, bn)) return WB_ECUDA;
    GemmParams p = base_params();
    p.M = N_FRAMES;
    p.N = D;
    p.batch = batch;
    for (int j = 0; j < 3; ++j)
      p.pass[j] = GemmPass{0, 0, static_cast<int8_t>(j), static_cast<int8_t>(j), 0, 0,
                           static_cast<int16_t>((C + 63) / 64), 0};
    p.n_pass = 3;
    // y1 rows go to rows 1..3000 of each item of y1p [batch][3001][D] (row 0 is the zero pad)
    if (!o_map(&g.omap, y1p, D, N_FRAMES + 1, batch, D, static_cast<uint64_t>(N_FRAMES + 1) * D)) return WB_ECUDA;
    p.out_row_off = 1;
    p.bias = w->conv1_b;
    g.p = p;
    Prof pr(PC_STEM_CONV1, s);
    WB_CUDA(launch_gemm(g, s));
  }
  {  // conv2: stride 2 -> one tensor map per tap over every other row of y1p
    GemmLaunch g;
    std::memset(&g, 0, sizeof(g));
    const int bn = D % 256 == 0 ? pick_bn(T_TOK, batch, D) : 128;
    g.bn = bn;
    g.epi = EPI_CONV2;
    const uint64_t rs = static_cast<uint64_t>(2 * D) * 2;
    for (int j = 0; j < 3; ++j)
      if (!a_map(&g.amap[j], false, y1p + static_cast<long long>(j) * D, D, T_TOK, 1, batch, rs, rs * T_TOK,
                 static_cast<uint64_t>(N_FRAMES + 1) * D * 2))
        return WB_ECUDA;
    g.amap[3] = g.amap[0];
    if (!b_map(&g.bmap, false, w->conv2_w, D, D, 3, static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(D) * D * 2,
               bn))
      return WB_ECUDA;
    GemmParams p = base_params();
    p.M = T_TOK;
    p.N = D;
    p.batch = batch;
    for (int j = 0; j < 3; ++j)
      p.pass[j] = GemmPass{static_cast<int8_t>(j), 0, 0, static_cast<int8_t>(j), 0, 0, static_cast<int16_t>(D / 64), 0};
    p.n_pass = 3;
    if (!o_map(&g.omap, x0, D, T_TOK, batch, D, static_cast<uint64_t>(T_TOK) * D)) return WB_ECUDA;
    p.bias = w->conv2_b;
    p.pos = pos;
    g.p = p;
    Prof pr(PC_STEM_CONV2, s);
    WB_CUDA(launch_gemm(g, s));
  }
  return WB_OK;
}

// -------------------------------- encoder ----------------------------------
size_t wb_encoder_workspace_bytes(const wb_dims* dims, int batch, const wb_precision* precision) {
  if (!dims_ok(dims) || batch < 1) return 0;
  return enc_layout(dims, batch, precision).total;
}

wb_status wb_encoder_forward(const void* x0, int batch, const wb_dims* dims, const wb_layer_weights* layers,
                             const wb_ln_weights* ln_post, const wb_precision* precision, int layer_begin,
                             int layer_end, int apply_final_ln, void* out, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!dims_ok(dims) || batch < 0 || layer_begin < 0 || layer_end < layer_begin || layer_end > dims->n_layers)
    return WB_EINVAL;
  wb_precision pr = {WB_BF16, WB_BF16, WB_BF16, WB_BF16, WB_BF16, WB_BF16};
  if (precision) pr = *precision;
  if (!site_ok(pr.qkv_w, pr.qkv_a) || !site_ok(pr.out_w, pr.out_a) || !site_ok(pr.ffn_w, pr.ffn_a))
    return WB_EUNSUPPORTED;
  if (batch == 0) return WB_OK;
  if (!x0 || !out || !aligned16(x0) || !aligned16(out) || x0 == out) return WB_EINVAL;
  if (layer_end > layer_begin && !layers) return WB_EINVAL;
  if (apply_final_ln && (!ln_post || !ln_post->g || !ln_post->b)) return WB_EINVAL;
  for (int l = layer_begin; l < layer_end; ++l) {
    const wb_layer_weights& L = layers[l];
    if (!L.ln1_g || !L.ln1_b || !L.w_qkv || !L.b_qkv || !L.w_out || !L.b_out || !L.ln2_g || !L.ln2_b || !L.w_fc1 ||
        !L.b_fc1 || !L.w_fc2 || !L.b_fc2)
      return WB_EINVAL;
    if ((pr.qkv_w == WB_E4M3 && !L.s_qkv) || (pr.out_w == WB_E4M3 && !L.s_out) ||
        (pr.ffn_w == WB_E4M3 && (!L.s_fc1 || !L.s_fc2)))
      return WB_EINVAL;
  }
  const EncLayout EL = enc_layout(dims, batch, &pr);
  if (!workspace || !aligned16(workspace) || workspace_bytes < EL.total) return WB_EWORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int D = dims->d_model, F = dims->d_ffn, H = dims->n_heads;
  const int M = batch * T_TOK;
  auto* h = reinterpret_cast<__nv_bfloat16*>(ws + EL.h);
  auto* a = reinterpret_cast<__nv_bfloat16*>(ws + EL.a);
  auto* qk = reinterpret_cast<__nv_bfloat16*>(ws + EL.qk);
  auto* vt = reinterpret_cast<__half*>(ws + EL.vt);
  auto* o = reinterpret_cast<__nv_bfloat16*>(ws + EL.o);
  auto* g = reinterpret_cast<__nv_bfloat16*>(ws + EL.g);
  auto* aq = EL.aq || pr.qkv_a == WB_E4M3 || pr.out_a == WB_E4M3 || pr.ffn_a == WB_E4M3
                 ? reinterpret_cast<uint8_t*>(ws + EL.aq)
                 : nullptr;
  auto* gq = pr.ffn_a == WB_E4M3 ? reinterpret_cast<uint8_t*>(ws + EL.gq) : nullptr;
  auto* slots = reinterpret_cast<float*>(ws + EL.slots);
  auto* stats = reinterpret_cast<float2*>(ws + EL.stats);
  auto* ln_part = reinterpret_cast<float2*>(ws + EL.ln_part);
  const auto* x0b = static_cast<const __nv_bfloat16*>(x0);
  auto* outb = static_cast<__nv_bfloat16*>(out);
  const float eps = 1e-5f;
  const int n_layers_run = layer_end - layer_begin;

  if (n_layers_run > 0 && (pr.qkv_a == WB_E4M3 || pr.out_a == WB_E4M3 || pr.ffn_a == WB_E4M3))
    WB_CUDA(cudaMemsetAsync(slots, 0, sizeof(float) * 4 * dims->n_layers * batch, s));
  // a bf16 site whose LayerNorm is folded into its GEMM reads the row statistics instead of LN's output
  auto fold_qkv = [&](int l) {
    return pr.qkv_a == WB_BF16 && layers[l].w_qkv_ln && layers[l].c_qkv && layers[l].b_qkv_ln;
  };
  auto fold_fc1 = [&](int l) {
    return pr.ffn_a == WB_BF16 && layers[l].w_fc1_ln && layers[l].c_fc1 && layers[l].b_fc1_ln;
  };
  // A folded LayerNorm's statistics come from the residual GEMM that writes its input (out-projection
  // for LN2, the previous layer's FC2 for LN1): its epilogue leaves (mean, M2) per row and column
  // group and a short pass merges them, instead of a pass that reads the whole activation again.  The
  // first layer's LN1 reads the stem output with the statistics kernel.
  const bool stats_in_epi = D % 32 == 0;
  bool stats_ready = false;   // the previous FC2 has left the partial statistics of this layer's input
  auto merge_stats = [&]() -> cudaError_t {
    Prof pr(PC_ENC_LN, s);
    return launch_ln_merge(ln_part, M, D / 32, 32, eps, stats, s);
  };

  for (int l = layer_begin; l < layer_end; ++l) {
    const wb_layer_weights& W = layers[l];
    // per-item absmax of the E4M3 operands: each 30 s chunk's activation gets its own scale
    float* am_qkv = slots + (4 * l + 0) * batch;
    float* am_out = slots + (4 * l + 1) * batch;
    float* am_fc1 = slots + (4 * l + 2) * batch;
    float* am_fc2 = slots + (4 * l + 3) * batch;
    const __nv_bfloat16* src = (l == layer_begin) ? x0b : h;
    const bool last = (l == layer_end - 1);
    const bool q8 = pr.qkv_a == WB_E4M3, o8 = pr.out_a == WB_E4M3, f8 = pr.ffn_a == WB_E4M3;

    const bool fq = fold_qkv(l), ff = fold_fc1(l);
    // LN1 -> a  [-> E4M3]  (folded: only the row statistics; QKV reads src itself)
    {
      if (fq && stats_ready) {
        WB_CUDA(merge_stats());
      } else if (fq) {
        Prof pr(PC_ENC_LN, s);
        WB_CUDA(launch_ln_stats(src, M, D, eps, stats, s));
      } else if (q8) {
        Prof pr(PC_ENC_LN, s, 2);   // E4M3 operand: LayerNorm writes the codes itself
        WB_CUDA(launch_layernorm_e4m3(src, W.ln1_g, W.ln1_b, M, D, eps, stats, am_qkv, T_TOK, aq, s));
      } else {
        Prof pr(PC_ENC_LN, s);
        WB_CUDA(launch_layernorm(src, nullptr, W.ln1_g, W.ln1_b, M, D, eps, a, nullptr, s));
      }
    }
    {  // QKV projection: q | k to qk [M, 2D], v transposed to vt
      GemmParams p = base_params();
      p.bias = W.b_qkv;
      p.vt = vt;
      p.vt_col0 = 2 * D;
      p.vt_T = T_TOK;
      p.vt_ld = T_PAD;
      p.vt_elems = static_cast<long long>(batch) * H * 64 * T_PAD;
      if (q8) {
        p.amax_a = am_qkv;
        p.scale_b = W.s_qkv;
      }
      const void* qkv_a = q8 ? static_cast<const void*>(aq) : static_cast<const void*>(a);
      const void* qkv_w = W.w_qkv;
      if (fq) {
        p.bias = W.b_qkv_ln;
        p.ln_stats = stats;
        p.ln_c = W.c_qkv;
        qkv_a = src;
        qkv_w = W.w_qkv_ln;
      }
      wb_status st = dense_gemm(qkv_a, qkv_w, M, 3 * D, D, q8, EPI_BIAS, qk, 2 * D, 2 * D, nullptr, p, s, PC_ENC_QKV);
      if (st != WB_OK) return st;
    }
    {
      // an E4M3 out-projection operand takes its per-chunk absmax from the attention epilogue
      wb_status st = run_attention(qk, qk + D, 2 * D, vt, batch, T_TOK, H, o, s, o8 ? am_out : nullptr);
      if (st != WB_OK) return st;
    }
    if (o8) {
      Prof pr(PC_ENC_QUANT, s);
      WB_CUDA(launch_quantize_rows(o, static_cast<long long>(M) * D, D, T_TOK, am_out, aq, s));
    }
    const bool ln2_in_epi = ff && stats_in_epi;
    {  // out projection + bias + residual -> h
      GemmParams p = base_params();
      p.bias = W.b_out;
      if (o8) {
        p.amax_a = am_out;
        p.scale_b = W.s_out;
      }
      if (ln2_in_epi) p.ln_part = ln_part;
      wb_status st = dense_gemm(o8 ? static_cast<const void*>(aq) : o, W.w_out, M, D, D, o8, EPI_BIAS_RESID, h, D, D,
                                src, p, s, PC_ENC_OUT);
      if (st != WB_OK) return st;
    }
    // LN2 -> a [-> E4M3]  (folded: only the row statistics; FC1 reads h itself)
    if (ff) {
      if (ln2_in_epi) {
        WB_CUDA(merge_stats());
      } else {
        Prof pr(PC_ENC_LN, s);
        WB_CUDA(launch_ln_stats(h, M, D, eps, stats, s));
      }
    } else if (f8) {
      Prof pr(PC_ENC_LN, s, 2);
      WB_CUDA(launch_layernorm_e4m3(h, W.ln2_g, W.ln2_b, M, D, eps, stats, am_fc1, T_TOK, aq, s));
    } else {
      Prof pr(PC_ENC_LN, s);
      WB_CUDA(launch_layernorm(h, nullptr, W.ln2_g, W.ln2_b, M, D, eps, a, nullptr, s));
    }
    {  // FC1 + bias + GELU -> g
      GemmParams p = base_params();
      p.bias = W.b_fc1;
      if (f8) {
        p.amax_a = am_fc1;
        p.scale_b = W.s_fc1;
        p.amax = am_fc2;
      }
      const void* fc1_a = f8 ? static_cast<const void*>(aq) : static_cast<const void*>(a);
      const void* fc1_w = W.w_fc1;
      if (ff) {
        p.bias = W.b_fc1_ln;
        p.ln_stats = stats;
        p.ln_c = W.c_fc1;
        fc1_a = h;
        fc1_w = W.w_fc1_ln;
      }
      wb_status st = dense_gemm(fc1_a, fc1_w, M, F, D, f8, EPI_BIAS_GELU, g, F, F, nullptr, p, s, PC_ENC_FC1);
      if (st != WB_OK) return st;
    }
    if (f8) {
      Prof pr(PC_ENC_QUANT, s);
      WB_CUDA(launch_quantize_rows(g, static_cast<long long>(M) * F, F, T_TOK, am_fc2, gq, s));
    }
    {  // FC2 + bias + residual -> h (or straight to out after the last layer without final LN)
      GemmParams p = base_params();
      p.bias = W.b_fc2;
      if (f8) {
        p.amax_a = am_fc2;
        p.scale_b = W.s_fc2;
      }
      void* dst = (last && !apply_final_ln) ? static_cast<void*>(outb) : static_cast<void*>(h);
      stats_ready = !last && fold_qkv(l + 1) && stats_in_epi;
      if (stats_ready) p.ln_part = ln_part;
      wb_status st = dense_gemm(f8 ? static_cast<const void*>(gq) : g, W.w_fc2, M, D, F, f8, EPI_BIAS_RESID, dst, D, D,
                                h, p, s, PC_ENC_FC2);
      if (st != WB_OK) return st;
    }
  }
  const __nv_bfloat16* final_src = n_layers_run > 0 ? h : x0b;
  if (apply_final_ln) {
    Prof pr(PC_ENC_LN, s);
    WB_CUDA(launch_layernorm(final_src, nullptr, ln_post->g, ln_post->b, M, D, eps, outb, nullptr, s));
  } else if (n_layers_run == 0) {
    WB_CUDA(cudaMemcpyAsync(outb, x0b, static_cast<size_t>(M) * D * 2, cudaMemcpyDeviceToDevice, s));
  }
  return WB_OK;
}

// --------------------------------- FP8 --------------------------------------
wb_status wb_quantize_fp8(const void* x, int64_t n, uint8_t* q, float* scale, void* stream) {
  if (n < 0 || !scale) return WB_EINVAL;
  if (n > 0 && (!x || !q || !aligned16(x) || !aligned16(q))) return WB_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  WB_CUDA(cudaMemsetAsync(scale, 0, sizeof(float), s));
  if (n > 0) {
    WB_CUDA(launch_amax(xb, n, scale, s));
    WB_CUDA(launch_quantize(xb, n, q, scale, nullptr, s));
  }
  WB_CUDA(launch_finalize_scale(scale, s));
  return WB_OK;
}

wb_status wb_dequantize_fp8(const uint8_t* q, const float* scale, int64_t n, void* y, void* stream) {
  if (n < 0 || !scale) return WB_EINVAL;
  if (n == 0) return WB_OK;
  if (!q || !y) return WB_EINVAL;
  WB_CUDA(launch_dequantize(q, scale, n, static_cast<__nv_bfloat16*>(y), static_cast<cudaStream_t>(stream)));
  return WB_OK;
}

wb_status wb_fold_layernorm(const void* w, const float* b, const float* gamma, const float* beta, int n_out, int d,
                            void* w_ln, float* c, float* b_ln, void* stream) {
  if (n_out < 0 || d <= 0 || d % 8) return WB_EINVAL;
  if (n_out == 0) return WB_OK;
  if (!w || !gamma || !beta || !w_ln || !c || !b_ln) return WB_EINVAL;
  if (!aligned16(w) || !aligned16(w_ln) || !aligned16(gamma) || !aligned16(beta) || (b && !aligned16(b)) ||
      !aligned16(c) || !aligned16(b_ln))
    return WB_EINVAL;
  WB_CUDA(launch_fold_ln(static_cast<const __nv_bfloat16*>(w), b, gamma, beta, n_out, d,
                         static_cast<__nv_bfloat16*>(w_ln), c, b_ln, static_cast<cudaStream_t>(stream)));
  return WB_OK;
}

// ------------------------------ building blocks ------------------------------
wb_status wb_linear(const void* a, const void* w, int M, int N, int K, int dtype, const float* bias,
                    const float* scale_a, const float* scale_w, int gelu, const void* resid, void* out,
                    void* stream) {
  if (M < 0 || N < 32 || N % 32 != 0 || K < 1) return WB_EINVAL;
  if (dtype != WB_BF16 && dtype != WB_E4M3) return WB_EUNSUPPORTED;
  const bool fp8 = dtype == WB_E4M3;
  if ((fp8 && K % 16 != 0) || (!fp8 && K % 8 != 0)) return WB_EINVAL;
  if (M == 0) return WB_OK;
  if (!a || !w || !out || !aligned16(a) || !aligned16(w) || !aligned16(out)) return WB_EINVAL;
  if (resid && !aligned16(resid)) return WB_EINVAL;
  if (fp8 && (!scale_a || !scale_w)) return WB_EINVAL;
  GemmParams p = base_params();
  p.bias = bias;
  p.act_gelu = gelu ? 1 : 0;
  if (fp8) {
    p.scale_a = scale_a;
    p.scale_b = scale_w;
  }
  const int epi = resid ? EPI_BIAS_RESID : gelu ? EPI_BIAS_GELU : EPI_BIAS;
  return dense_gemm(a, w, M, N, K, fp8, epi, out, N, N, resid, p, static_cast<cudaStream_t>(stream));
}

wb_status wb_layernorm(const void* x, const void* residual, const float* g, const float* b, int rows, int d,
                       float eps, void* y, void* total, void* stream) {
  if (rows < 0 || d < 128 || d > 2048 || d % 128 != 0 || !(eps > 0.0f)) return WB_EINVAL;
  if (rows == 0) return WB_OK;
  if (!x || !g || !b || !y || !aligned16(x) || !aligned16(y) || !aligned16(g) || !aligned16(b)) return WB_EINVAL;
  if ((residual && !aligned16(residual)) || (total && (!residual || !aligned16(total)))) return WB_EINVAL;
  WB_CUDA(launch_layernorm(static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(residual), g, b,
                           rows, d, eps, static_cast<__nv_bfloat16*>(y), static_cast<__nv_bfloat16*>(total),
                           static_cast<cudaStream_t>(stream)));
  return WB_OK;
}

wb_status wb_layernorm_e4m3(const void* x, const float* g, const float* b, int rows, int d, float eps,
                            int rows_per_item, uint8_t* q, float* amax, float* stats, void* stream) {
  if (rows < 0 || d < 128 || d > 2048 || d % 128 != 0 || !(eps > 0.0f) || rows_per_item < 1) return WB_EINVAL;
  if (rows == 0) return WB_OK;
  if (!x || !g || !b || !q || !amax || !stats || !aligned16(x) || !aligned16(g) || !aligned16(b) || !aligned16(q) ||
      !aligned16(stats) || (reinterpret_cast<uintptr_t>(amax) & 3u))
    return WB_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int items = (rows + rows_per_item - 1) / rows_per_item;
  WB_CUDA(cudaMemsetAsync(amax, 0, sizeof(float) * items, s));
  WB_CUDA(launch_layernorm_e4m3(static_cast<const __nv_bfloat16*>(x), g, b, rows, d, eps,
                                reinterpret_cast<float2*>(stats), amax, rows_per_item, q, s));
  return WB_OK;
}

size_t wb_attention_workspace_bytes(int batch, int T, int n_heads) {
  if (batch < 1 || T < 1 || n_heads < 1) return 0;
  return static_cast<size_t>(batch) * n_heads * 64 * T_PAD * 2;
}

wb_status wb_attention(const void* q, const void* k, const void* v, int batch, int T, int n_heads, void* out,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (batch < 0 || T < 1 || T > T_PAD || n_heads < 1 || n_heads > 32) return WB_EINVAL;
  if (batch == 0) return WB_OK;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return WB_EINVAL;
  if (!workspace || !aligned16(workspace) || workspace_bytes < wb_attention_workspace_bytes(batch, T, n_heads))
    return WB_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* vt = static_cast<__half*>(workspace);
  const long long d = 64LL * n_heads;
  WB_CUDA(launch_transpose_v(static_cast<const __nv_bfloat16*>(v), d, batch, T, n_heads, vt, s));
  return run_attention(static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), d, vt, batch, T,
                       n_heads, static_cast<__nv_bfloat16*>(out), s);
}

// -------------------------- decoder-side / extra building blocks --------------------------
wb_status wb_rmsnorm(const void* x, const void* residual, const float* g, int rows, int d, float eps, void* y,
                     void* total, void* stream) {
  if (rows < 0 || d < 128 || d > 2048 || d % 128 != 0 || !(eps > 0.0f)) return WB_EINVAL;
  if (rows == 0) return WB_OK;
  if (!x || !g || !y || !aligned16(x) || !aligned16(y) || !aligned16(g)) return WB_EINVAL;
  if ((residual && !aligned16(residual)) || (total && (!residual || !aligned16(total)))) return WB_EINVAL;
  WB_CUDA(launch_rmsnorm(static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(residual), g, rows,
                         d, eps, static_cast<__nv_bfloat16*>(y), static_cast<__nv_bfloat16*>(total),
                         static_cast<cudaStream_t>(stream)));
  return WB_OK;
}

wb_status wb_quantize_e5m2(const void* x, int64_t n, uint8_t* q, float* scale, void* stream) {
  if (n < 0 || !scale) return WB_EINVAL;
  if (n > 0 && (!x || !q || !aligned16(x))) return WB_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  WB_CUDA(cudaMemsetAsync(scale, 0, sizeof(float), s));
  if (n > 0) WB_CUDA(launch_amax(xb, n, scale, s));
  WB_CUDA(launch_quantize_e5m2(xb, n, q, scale, s));
  return WB_OK;
}

wb_status wb_dequantize_e5m2(const uint8_t* q, const float* scale, int64_t n, void* y, void* stream) {
  if (n < 0 || !scale) return WB_EINVAL;
  if (n == 0) return WB_OK;
  if (!q || !y) return WB_EINVAL;
  WB_CUDA(launch_dequantize_e5m2(q, scale, n, static_cast<__nv_bfloat16*>(y), static_cast<cudaStream_t>(stream)));
  return WB_OK;
}

wb_status wb_cross_kv(const void* enc_out, int batch, const wb_dims* dims, int n_dec_layers,
                      const wb_cross_kv_weights* w, void* kv, void* stream) {
  if (!dims_ok(dims) || batch < 0 || n_dec_layers < 0) return WB_EINVAL;
  if (batch == 0 || n_dec_layers == 0) return WB_OK;
  if (!enc_out || !w || !kv || !aligned16(enc_out) || !aligned16(kv)) return WB_EINVAL;
  const int D = dims->d_model, M = batch * T_TOK;
  for (int l = 0; l < n_dec_layers; ++l)
    if (!w[l].w_kv || !w[l].b_kv || !aligned16(w[l].w_kv)) return WB_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int l = 0; l < n_dec_layers; ++l) {
    GemmParams p = base_params();
    p.bias = w[l].b_kv;
    void* out = static_cast<__nv_bfloat16*>(kv) + static_cast<size_t>(l) * M * 2 * D;
    const wb_status st = dense_gemm(enc_out, w[l].w_kv, M, 2 * D, D, false, EPI_BIAS, out, 2 * D, 2 * D, nullptr, p,
                                    s, PC_OTHER);
    if (st != WB_OK) return st;
  }
  return WB_OK;
}

// -------------------------------- profiling ----------------------------------
wb_status wb_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& r : g_prof_recs) {
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_recs.clear();
  g_prof_on = true;
  return WB_OK;
}

int wb_profile_end(int max_classes, const char** names, double* total_ms, int64_t* launches) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof_on = false;
  double ms[PC_COUNT] = {0};
  int64_t cnt[PC_COUNT] = {0};
  for (auto& r : g_prof_recs) {
    float t = 0.0f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) ms[r.cls] += t;
    cnt[r.cls] += r.kernels;
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_recs.clear();
  const int n = max_classes < PC_COUNT ? max_classes : PC_COUNT;
  for (int i = 0; i < n; ++i) {
    if (names) names[i] = kProfNames[i];
    if (total_ms) total_ms[i] = ms[i];
    if (launches) launches[i] = cnt[i];
  }
  return PC_COUNT;
}

}  // extern "C"
