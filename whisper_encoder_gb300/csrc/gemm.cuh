// Persistent tcgen05 GEMM for sm_103a: D[b, m, n] = sum_passes sum_k A_p[b, m, k] * B_p[n, k].
//
// One kernel family carries every dense contraction of the hot path (the
// whisper-blaze showcase site, "The Solution", gemm_hopper.cu card: a TMA-fed
// asynchronous tensor-core GEMM; here rebuilt on tcgen05 with TMEM
// accumulators instead of Hopper warpgroup MMA):
//   * QKV / out-projection / FC1 / FC2 (bf16 or E4M3 operands),
//   * the conv stem as an implicit GEMM (one pass per kernel tap),
//   * the windowed real DFT and the mel filterbank (split-bf16 passes).
//
// Roles (192 threads): warp 0 lane 0 issues TMA loads into a ring of smem
// stages; warp 1 lane 0 issues tcgen05.mma into one of two TMEM accumulators;
// warps 2-5 (128 threads, one accumulator row each) run the epilogue of tile
// i while the MMA warp already accumulates tile i+1.  All waits are bounded.
//
// K schedule: a list of passes; pass p reads A through tensor map amap[p]
// (4-D: k, row, part, batch) at row offset a_row_off and part a_part, and B
// through bmap (3-D: k, n, part) at part b_part, with n_kb blocks of BK
// elements starting at k offsets a_x0 / b_x0.
#pragma once
#include "ptx.cuh"
#include "types.h"

namespace wb {

template <int BN>
struct GemmSmem {
  static constexpr int A_BYTES = GEMM_BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int BAR_BYTES = 256;
  static constexpr int TOTAL = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
};

__device__ __forceinline__ float sinusoid(int t, int n, int d) {
  const int half = d >> 1;
  const int i = n < half ? n : n - half;
  const float inc = 9.210340371976184f / static_cast<float>(half - 1);  // ln(10000) / (d/2 - 1)
  const float ang = static_cast<float>(t) * expf(-inc * static_cast<float>(i));
  return n < half ? sinf(ang) : cosf(ang);
}

template <int BN, bool FP8, int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap amap0, const __grid_constant__ CUtensorMap amap1,
                const __grid_constant__ CUtensorMap amap2, const __grid_constant__ CUtensorMap amap3,
                const __grid_constant__ CUtensorMap bmap, const __grid_constant__ GemmParams p) {
  using S = GemmSmem<BN>;
  constexpr int STAGES = S::STAGES;
  constexpr uint32_t IDESC = make_idesc(GEMM_BM, BN, FP8 ? 0u : 1u);
  constexpr int KSTEPS = 4;  // 128-byte rows: 4 x K16 (bf16) or 4 x K32 (E4M3)
  constexpr int BK = FP8 ? 128 : 64;
  constexpr uint32_t TMEM_COLS = 2 * BN;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_u32 - smem_u32(smem_raw));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES);
  uint64_t* full = bars;                 // [STAGES]
  uint64_t* empty = bars + STAGES;       // [STAGES]
  uint64_t* tfull = bars + 2 * STAGES;   // [2]
  uint64_t* tempty = tfull + 2;          // [2]
  uint64_t* mma_done = tempty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id();
  const int lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int m_tiles = (p.M + GEMM_BM - 1) / GEMM_BM;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tiles_per_item = m_tiles * n_tiles;
  const int total_tiles = tiles_per_item * p.batch;
  int n_iter = 0;
  for (int q = 0; q < p.n_pass; ++q) n_iter += p.pass[q].n_kb;

  if (warp == 0) {
    // ------------------------------ TMA producer ---------------------------
    if (lane == 0) {
      tma_prefetch_desc(&amap0);
      tma_prefetch_desc(&bmap);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_parity = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const int b = tile / tiles_per_item;
        const int r = tile % tiles_per_item;
        const int mt = r / n_tiles, nt = r % n_tiles;
        for (int q = 0; q < p.n_pass && ok; ++q) {
          const GemmPass ps = p.pass[q];
          const CUtensorMap* am = ps.amap == 0 ? &amap0 : ps.amap == 1 ? &amap1 : ps.amap == 2 ? &amap2 : &amap3;
          for (int kb = 0; kb < ps.n_kb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, p.err, abort_flag, 1)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[stage], S::STAGE_BYTES);
            uint8_t* sa = smem + stage * S::STAGE_BYTES;
            uint8_t* sb = sa + S::A_BYTES;
            tma_load_4d(sa, am, &full[stage], ps.a_x0 + kb * BK, mt * GEMM_BM + ps.a_row_off, ps.a_part, b);
            tma_load_3d(sb, &bmap, &full[stage], ps.b_x0 + kb * BK, nt * BN, ps.b_part);
            issued_mask |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
      if (!ok) {  // let every copy already in flight land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s)) mbar_drain(&full[s], (last_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer -----------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.err, abort_flag, 2)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int it = 0; it < n_iter; ++it) {
          if (!mbar_wait(&full[stage], phase, p.err, abort_flag, 3)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          const uint32_t sb = sa + S::A_BYTES;
#pragma unroll
          for (int k = 0; k < KSTEPS; ++k) {
            const uint64_t ad = sw128_desc(sa + k * 32);
            const uint64_t bd = sw128_desc(sb + k * 32);
            if (FP8)
              mma_e4m3(d_tmem, ad, bd, IDESC, (it | k) != 0);
            else
              mma_bf16(d_tmem, ad, bd, IDESC, (it | k) != 0);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (ok) mma_commit(&tfull[acc]);
      }
      // make sure no MMA is still reading smem or writing TMEM when the CTA leaves
      mma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // ------------------------------- epilogue ------------------------------
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int row_in_tile = quarter * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait(&tfull[acc], acc_phase, p.err, abort_flag, 4)) break;
      tc_fence_after();
      const int b = tile / tiles_per_item;
      const int r = tile % tiles_per_item;
      const int mt = r / n_tiles, nt = r % n_tiles;
      const int m = mt * GEMM_BM + row_in_tile;
      const bool row_ok = m < p.M;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;

      if constexpr (EPI == EPI_STD) {
        float alpha = 1.0f;
        if (p.scale_a) alpha *= *p.scale_a;
        if (p.scale_b) alpha *= *p.scale_b;
        float local_amax = 0.0f;
        const long long orow = static_cast<long long>(b) * p.out_batch_rows + p.out_row_off + m;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int n0 = nt * BN + c * 32;
          if (n0 >= p.N) break;
          float v[32];
          tmem_ld32(t_row + c * 32, v);
          tmem_ld_wait();
          if (!row_ok) continue;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x = v[i] * alpha;
            if (p.bias) x += __ldg(p.bias + n0 + i);
            if (p.act_gelu) x = gelu_erf(x);
            if (p.add_pe) x += sinusoid(m, n0 + i, p.N);
            v[i] = x;
          }
          if (p.vt && n0 >= p.vt_col0) {
            // V goes out transposed: row (b*H + h)*64 + e, column t
            const int col = n0 - p.vt_col0;
            const int gb = (b * p.M + m) / p.vt_T, t = (b * p.M + m) % p.vt_T;
            const int h = col >> 6, e0 = col & 63;
            const int H = (p.N - p.vt_col0) >> 6;
            __nv_bfloat16* dst = p.vt + (static_cast<long long>(gb * H + h) * 64 + e0) * p.vt_ld + t;
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[static_cast<long long>(i) * p.vt_ld] = __float2bfloat16_rn(v[i]);
            continue;
          }
          if (p.resid) {
            const uint4* rp = reinterpret_cast<const uint4*>(p.resid + orow * p.ldo + n0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 u = rp[j];
              const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
              for (int i = 0; i < 8; ++i) v[j * 8 + i] += __bfloat162float(hv[i]);
            }
          }
          uint4 pk[4];
          uint32_t* pw32 = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
          for (int i = 0; i < 16; ++i) pw32[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
          if (p.amax) {
            const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(pk);
#pragma unroll
            for (int i = 0; i < 32; ++i) local_amax = fmaxf(local_amax, fabsf(__bfloat162float(hv[i])));
          }
          uint4* op = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * p.ldo + n0);
#pragma unroll
          for (int j = 0; j < 4; ++j) op[j] = pk[j];
        }
        if (p.amax) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) local_amax = fmaxf(local_amax, __shfl_xor_sync(0xffffffffu, local_amax, o));
          if (lane == 0 && local_amax > 0.0f) atomic_max_nonneg(p.amax, local_amax);
        }
      } else if constexpr (EPI == EPI_POWER) {
        // columns [0, BN/2) hold the cosine part and [BN/2, BN) the sine part of the same bins
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          float re[32], im[32];
          tmem_ld32(t_row + c * 32, re);
          tmem_ld32(t_row + BN / 2 + c * 32, im);
          tmem_ld_wait();
          if (!row_ok) continue;
          const int bin0 = nt * (BN / 2) + c * 32;
          uint4 hi[4], lo[4];
          uint32_t* h32 = reinterpret_cast<uint32_t*>(hi);
          uint32_t* l32 = reinterpret_cast<uint32_t*>(lo);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = re[2 * i] * re[2 * i] + im[2 * i] * im[2 * i];
            const float p1 = re[2 * i + 1] * re[2 * i + 1] + im[2 * i + 1] * im[2 * i + 1];
            const __nv_bfloat16 a0 = __float2bfloat16_rn(p0), a1 = __float2bfloat16_rn(p1);
            h32[i] = pack_bf16(__bfloat162float(a0), __bfloat162float(a1));
            l32[i] = pack_bf16(p0 - __bfloat162float(a0), p1 - __bfloat162float(a1));
          }
          const long long rowi = static_cast<long long>(b) * 2 * p.M + m;
          uint4* dh = reinterpret_cast<uint4*>(p.pw + rowi * p.pw_ld + bin0);
          uint4* dl = reinterpret_cast<uint4*>(p.pw + (rowi + p.M) * p.pw_ld + bin0);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            dh[j] = hi[j];
            dl[j] = lo[j];
          }
        }
      } else {  // EPI_MEL
        float local_max = 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int n0 = nt * BN + c * 32;
          float v[32];
          tmem_ld32(t_row + c * 32, v);
          tmem_ld_wait();
          if (!row_ok || n0 >= p.n_valid) continue;
          float* dst = p.mel_out + (static_cast<long long>(b) * p.n_valid + n0) * p.M + m;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (n0 + i < p.n_valid) {
              const float mv = v[i] > 0.0f ? v[i] : 0.0f;
              local_max = fmaxf(local_max, mv);
              dst[static_cast<long long>(i) * p.M] = log10f(fmaxf(mv, 1e-10f));
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) local_max = fmaxf(local_max, __shfl_xor_sync(0xffffffffu, local_max, o));
        if (lane == 0 && local_max > 0.0f) atomic_max_nonneg(p.mel_max + b, local_max);
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace wb
