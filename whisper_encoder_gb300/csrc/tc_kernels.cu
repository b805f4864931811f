// Instantiation and launch of the tensor-core kernels (GEMM family, attention).
#include <mutex>

#include "internal.h"
#include "gemm.cuh"
#include "attention.cuh"

namespace wb {

namespace {

constexpr int kMaxDev = 64;
int g_sm_count[kMaxDev] = {0};
std::mutex g_attr_mu;

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return (dev >= 0 && dev < kMaxDev) ? dev : 0;
}

// Raise a kernel's dynamic shared-memory limit once per device (so that launches stay free of
// attribute calls, which keeps them legal inside CUDA-graph stream capture).
template <typename K>
cudaError_t ensure_smem_attr(K kern, int smem, uint64_t* done_mask) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (*done_mask & (1ull << dev)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) *done_mask |= 1ull << dev;
  return e;
}

}  // namespace

int sm_count() {
  const int dev = current_device();
  if (g_sm_count[dev] <= 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = n > 0 ? n : 1;
  }
  return g_sm_count[dev];
}

namespace {

template <int BN, bool FP8, int EPI>
cudaError_t gemm_launch_t(const GemmLaunch& g, cudaStream_t s) {
  auto kern = gemm_kernel<BN, FP8, EPI>;
  const int smem = GemmSmem<BN>::TOTAL;
  static uint64_t attr_done = 0;
  cudaError_t e = ensure_smem_attr(kern, smem, &attr_done);
  if (e != cudaSuccess) return e;
  const int m_tiles = (g.p.M + GEMM_BM - 1) / GEMM_BM;
  const int n_tiles = (g.p.N + BN - 1) / BN;
  const long long tiles = static_cast<long long>(m_tiles) * n_tiles * g.p.batch;
  int grid = sm_count();
  if (tiles < grid) grid = static_cast<int>(tiles);
  if (grid < 1) return cudaSuccess;
  return launch_pdl(kern, dim3(grid), dim3(GEMM_THREADS), smem, s, g.amap[0], g.amap[1], g.amap[2], g.amap[3], g.bmap,
                    g.omap, g.p);
}

}  // namespace

cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t s) {
#define WB_GEMM_STD(BN)                                                                                        \
  switch (g.epi) {                                                                                             \
    case EPI_BIAS: return g.fp8 ? gemm_launch_t<BN, true, EPI_BIAS>(g, s) : gemm_launch_t<BN, false, EPI_BIAS>(g, s); \
    case EPI_BIAS_GELU:                                                                                        \
      return g.fp8 ? gemm_launch_t<BN, true, EPI_BIAS_GELU>(g, s) : gemm_launch_t<BN, false, EPI_BIAS_GELU>(g, s); \
    case EPI_BIAS_RESID:                                                                                       \
      return g.fp8 ? gemm_launch_t<BN, true, EPI_BIAS_RESID>(g, s) : gemm_launch_t<BN, false, EPI_BIAS_RESID>(g, s); \
    case EPI_CONV2:                                                                                            \
      if (!g.fp8) return gemm_launch_t<BN, false, EPI_CONV2>(g, s);                                           \
      break;                                                                                                   \
    default: break;                                                                                            \
  }
  if (g.bn == 256) {
    WB_GEMM_STD(256)
    if (g.epi == EPI_POWER && !g.fp8) return gemm_launch_t<256, false, EPI_POWER>(g, s);
  } else if (g.bn == 128) {
    WB_GEMM_STD(128)
    if (g.epi == EPI_MEL && !g.fp8) return gemm_launch_t<128, false, EPI_MEL>(g, s);
  }
#undef WB_GEMM_STD
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& vt,
                             const AttnParams& p, cudaStream_t s) {
  const int smem = AttnSmem::TOTAL;
  static uint64_t attr_done = 0;
  cudaError_t e = ensure_smem_attr(attention_kernel, smem, &attr_done);
  if (e != cudaSuccess) return e;
  const int n_qt = (p.T + ATT_BQ - 1) / ATT_BQ;
  const long long grid = static_cast<long long>(p.batch) * p.H * n_qt;
  if (grid < 1) return cudaSuccess;
  return launch_pdl(attention_kernel, dim3(static_cast<unsigned>(grid)), dim3(ATT_THREADS), smem, s, q, k, vt, p);
}

}  // namespace wb
