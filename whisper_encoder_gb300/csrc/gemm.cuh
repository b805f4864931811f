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
// Roles (576 threads): warp 0 lane 0 issues TMA loads into a ring of smem
// stages; warp 1 lane 0 issues tcgen05.mma into one of two TMEM accumulators;
// warps 2-17 run the epilogue of tile i while the MMA warp already
// accumulates tile i+1.  Epilogue warp w owns TMEM lane quarter w%4 (32 rows)
// and one quarter of the tile's columns; it stages its 32x32 output boxes in
// shared memory and writes them with TMA bulk stores.  The residual of the
// residual epilogue is read with plain 16-byte global loads, all of a thread's
// columns issued before the accumulator is ready.  All waits are bounded.
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
  static constexpr int EPI_BOX_BYTES = 32 * 64;   // one 32 x 32 bf16 box per epilogue warp (64-byte swizzle)
  static constexpr int OFF_EPI = STAGES * STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_EPI + GEMM_EPI_WARPS * EPI_BOX_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int TOTAL = 1024 + OFF_BAR + BAR_BYTES;
};

// Byte offset of 16-byte chunk j (columns 8j..8j+7) of row r in a 32 x 64-byte box stored with
// the 64-byte swizzle (chunk index XOR address bits 7-8), as TMA reads and writes it.
__device__ __forceinline__ uint32_t box_off(int r, int j) {
  return static_cast<uint32_t>(r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
}

template <int BN, bool FP8, int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap amap0, const __grid_constant__ CUtensorMap amap1,
                const __grid_constant__ CUtensorMap amap2, const __grid_constant__ CUtensorMap amap3,
                const __grid_constant__ CUtensorMap bmap, const __grid_constant__ CUtensorMap omap,
                const __grid_constant__ GemmParams p) {
  using S = GemmSmem<BN>;
  constexpr int STAGES = S::STAGES;
  constexpr uint32_t IDESC = make_idesc(GEMM_BM, BN, FP8 ? 0u : 1u);
  constexpr int KSTEPS = 4;  // 128-byte rows: 4 x K16 (bf16) or 4 x K32 (E4M3)
  constexpr int BK = FP8 ? 128 : 64;
  constexpr uint32_t TMEM_COLS = 2 * BN;
  constexpr bool STD = EPI == EPI_BIAS || EPI == EPI_BIAS_GELU || EPI == EPI_BIAS_RESID || EPI == EPI_CONV2;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_u32 - smem_u32(smem_raw));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* full = bars;                       // [STAGES]
  uint64_t* empty = bars + STAGES;             // [STAGES]
  uint64_t* tfull = bars + 2 * STAGES;         // [2]
  uint64_t* tempty = tfull + 2;                // [2]
  uint64_t* mma_done = tempty + 2;             // [1]
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
      mbar_init(&tempty[a], GEMM_EPI_WARPS);
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
  // barriers and TMEM are set up: from here on the kernel reads its inputs
  grid_dependency_wait();
  grid_dependents_launch();

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
    constexpr int COLS = BN / 4;                 // columns per epilogue warp
    constexpr int CHUNKS = COLS / 32;
    const int ew = warp - 2;                     // 0 .. GEMM_EPI_WARPS-1
    const int quarter = warp & 3;                // TMEM lane quarter this warp may access
    const int cg = ew >> 2;                      // column group
    uint8_t* box = smem + S::OFF_EPI + ew * S::EPI_BOX_BYTES;
    bool ok = true;
    int local = 0;
    float alpha_w = 1.0f, alpha_a = 1.0f;
    if (FP8) {
      if (p.scale_a) alpha_a = *p.scale_a;
      if (p.scale_b) alpha_w = *p.scale_b;
    }

    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const int b = tile / tiles_per_item;
      const int r = tile % tiles_per_item;
      const int mt = r / n_tiles, nt = r % n_tiles;
      const int m0 = mt * GEMM_BM + quarter * 32;      // first row of this warp's slab
      const int m = m0 + lane;
      const bool row_ok = m < p.M;
      const int ncol0 = nt * BN + cg * COLS;
      // residual of this thread's row: all CHUNKS x 32 columns (64 bytes each) loaded before the
      // accumulator is ready, so their latency hides behind the main loop
      uint4 rres[EPI == EPI_BIAS_RESID ? CHUNKS * 4 : 1];
      if constexpr (EPI == EPI_BIAS_RESID) {
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
          const int n0 = ncol0 + c * 32;
#pragma unroll
          for (int j = 0; j < 4; ++j) rres[4 * c + j] = make_uint4(0u, 0u, 0u, 0u);
          const long long ri = b * p.resid_item + static_cast<long long>(p.out_row_off + m) * p.resid_ld + n0;
          if (row_ok && n0 < p.N && in_bounds(p.err, ri, 32, p.resid_elems, SITE_GEMM_RESID)) {
            const uint4* rp = reinterpret_cast<const uint4*>(p.resid + ri);
#pragma unroll
            for (int j = 0; j < 4; ++j) rres[4 * c + j] = rp[j];
          }
        }
      }
      // folded LayerNorm: this row's (mean, rstd), fetched while the accumulator is still being computed
      const bool lnf = (EPI == EPI_BIAS || EPI == EPI_BIAS_GELU) && !FP8 && p.ln_stats != nullptr;
      float2 ln_mr = make_float2(0.0f, 1.0f);
      if (lnf && row_ok &&
          in_bounds(p.err, static_cast<long long>(b) * p.M + m, 1, static_cast<long long>(p.batch) * p.M,
                    SITE_GEMM_LNSTATS))
        ln_mr = p.ln_stats[static_cast<long long>(b) * p.M + m];
      if (!mbar_wait(&tfull[acc], acc_phase, p.err, abort_flag, 4)) { ok = false; break; }
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;

      if constexpr (STD) {
        // flattened row -> batch item (chunk) for the per-item E4M3 scales
        const int item = p.rows_per_item > 0 ? (b * p.M + (row_ok ? m : p.M - 1)) / p.rows_per_item : 0;
        float alpha = alpha_w * alpha_a;
        if (FP8 && p.amax_a) {
          const float am = in_bounds(p.err, item, 1, p.amax_items, SITE_GEMM_AMAX) ? __ldg(p.amax_a + item) : 0.0f;
          alpha = alpha_w * (am > 0.0f ? am / 448.0f : 1.0f);
        }
        float tile_amax = 0.0f;
        const float ln_mu = ln_mr.x, ln_rs = ln_mr.y;
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
          const int n0 = ncol0 + c * 32;
          float v[32];
          tmem_ld32(t_row + cg * COLS + c * 32, v);
          tmem_ld_wait();
          if (c == CHUNKS - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);     // accumulator is free for tile i+2
          }
          if (n0 >= p.N) continue;
          if (!in_bounds(p.err, n0, 32, p.N, SITE_GEMM_BIAS)) continue;

          // bias (+ E4M3 scale) and activation
          const float4* bp = reinterpret_cast<const float4*>(p.bias + n0);
          const float4* cp = reinterpret_cast<const float4*>(p.ln_c + n0);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 bb = p.bias ? __ldg(bp + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float bv[4] = {bb.x, bb.y, bb.z, bb.w};
            const float4 c4 = lnf ? __ldg(cp + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int kk = 0; kk < 4; kk += 2) {
              // two columns at a time with packed fp32 arithmetic
              float x0, x1;
              const uint64_t acc2 = f32x2_pack(v[4 * i4 + kk], v[4 * i4 + kk + 1]);
              const uint64_t b2 = f32x2_pack(bv[kk], bv[kk + 1]);
              if (lnf) {
                const uint64_t t2 = f32x2_fma(f32x2_pack(cv[kk], cv[kk + 1]), f32x2_pack(-ln_mu, -ln_mu), acc2);
                f32x2_unpack(f32x2_fma(f32x2_pack(ln_rs, ln_rs), t2, b2), x0, x1);
              } else if (FP8) {
                f32x2_unpack(f32x2_fma(acc2, f32x2_pack(alpha, alpha), b2), x0, x1);
              } else {
                f32x2_unpack(f32x2_fma(acc2, f32x2_pack(1.0f, 1.0f), b2), x0, x1);   // one rounding, as x + b
              }
              if (EPI == EPI_BIAS_GELU || EPI == EPI_CONV2 || (EPI == EPI_BIAS_RESID && p.act_gelu)) {
                // measured: the packed form is faster where the main loop bounds the tile (bf16) and
                // slower where the epilogue does (E4M3, twice the MMA rate)
                if (FP8) {
                  x0 = gelu_fast(x0);
                  x1 = gelu_fast(x1);
                } else {
                  gelu_fast_x2(x0, x1);
                }
              }
              if (EPI == EPI_CONV2) {   // positional embedding from the table (row m, this column pair)
                const int mr = row_ok ? m : p.M - 1;      // rows past M are not stored; stay inside the table
                const long long pi = static_cast<long long>(mr) * p.N + n0 + 4 * i4 + kk;
                const float2 pe = in_bounds(p.err, pi, 2, static_cast<long long>(p.M) * p.N, SITE_GEMM_POS)
                                      ? __ldg(reinterpret_cast<const float2*>(p.pos + pi))
                                      : make_float2(0.0f, 0.0f);
                x0 += pe.x;
                x1 += pe.y;
              }
              v[4 * i4 + kk] = x0;
              v[4 * i4 + kk + 1] = x1;
            }
          }
          if (EPI == EPI_BIAS && p.vt && n0 >= p.vt_col0) {
            // V goes out transposed: row (b*H + h)*64 + e, column t (32 lanes = 32 consecutive t)
            if (row_ok) {
              const int col = n0 - p.vt_col0;
              const int gb = m / p.vt_T, t = m % p.vt_T;
              const int h = col >> 6, e0 = col & 63;
              const int H = (p.N - p.vt_col0) >> 6;
              const long long di = (static_cast<long long>(gb * H + h) * 64 + e0) * p.vt_ld + t;
              __half* dst = p.vt + di;
              if (in_bounds(p.err, di, 31LL * p.vt_ld + 1, p.vt_elems, SITE_GEMM_VT)) {
#pragma unroll
                for (int i = 0; i < 32; ++i)   // f16 for the attention's f16 P.V product (saturated to its range)
                  dst[static_cast<long long>(i) * p.vt_ld] = __float2half_rn(fminf(fmaxf(v[i], -65504.0f), 65504.0f));
              }
            }
            continue;
          }
          if constexpr (EPI == EPI_BIAS_RESID) {
            // residual pairs: bf16 -> fp32 by shifts, added with packed fp32 pairs (one rounding each)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t rw[4] = {rres[4 * c + j].x, rres[4 * c + j].y, rres[4 * c + j].z, rres[4 * c + j].w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint64_t r2 = f32x2_pack(__uint_as_float(rw[i] << 16), __uint_as_float(rw[i] & 0xffff0000u));
                f32x2_unpack(f32x2_fma(f32x2_pack(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]), f32x2_pack(1.0f, 1.0f), r2),
                             v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
              }
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
          if (EPI == EPI_BIAS_RESID && p.ln_part && row_ok) {
            // the next LayerNorm's statistics: (mean, M2) of these 32 stored (bf16) outputs,
            // accumulated about the first of them (so that the sums do not cancel), for a pass that
            // merges each row's N / 32 groups once the whole output is written (the same groups at
            // every tile width)
            const float k0 = __uint_as_float(pk[0] << 16);
            const uint64_t one2 = f32x2_pack(1.0f, 1.0f), nk2 = f32x2_pack(-k0, -k0);
            uint64_t s1 = f32x2_pack(0.0f, 0.0f), s2 = s1;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint64_t d2 =
                  f32x2_fma(f32x2_pack(__uint_as_float(pk[i] << 16), __uint_as_float(pk[i] & 0xffff0000u)), one2, nk2);
              s1 = f32x2_fma(d2, one2, s1);
              s2 = f32x2_fma(d2, d2, s2);
            }
            float a0, a1, q0, q1;
            f32x2_unpack(s1, a0, a1);
            f32x2_unpack(s2, q0, q1);
            const float sd = a0 + a1;
            // group-major, so that a warp's 32 rows write 256 contiguous bytes
            const long long rows_all = static_cast<long long>(p.batch) * p.M;
            const long long pi = static_cast<long long>(n0 >> 5) * rows_all + static_cast<long long>(b) * p.M + m;
            if (in_bounds(p.err, pi, 1, rows_all * (p.N >> 5), SITE_GEMM_LNPART))
              p.ln_part[pi] = make_float2(k0 + sd * (1.0f / 32.0f), fmaxf((q0 + q1) - sd * sd * (1.0f / 32.0f), 0.0f));
          }
          if (lane == 0) bulk_wait_read0();       // the previous store has read the staging box
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(box + box_off(lane, j)) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&omap, box, n0, p.out_row_off + m0, b);
            bulk_commit();
          }
        }
        if (p.amax) {   // one atomic per warp and tile; per lane where the 32 rows straddle two chunks
          const int item0 = __shfl_sync(0xffffffffu, item, 0);
          if (__all_sync(0xffffffffu, item == item0)) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tile_amax = fmaxf(tile_amax, __shfl_xor_sync(0xffffffffu, tile_amax, o));
            if (lane == 0 && tile_amax > 0.0f && in_bounds(p.err, item0, 1, p.amax_items, SITE_GEMM_AMAX))
              atomic_max_nonneg(p.amax + item0, tile_amax);
          } else if (tile_amax > 0.0f && in_bounds(p.err, item, 1, p.amax_items, SITE_GEMM_AMAX)) {
            atomic_max_nonneg(p.amax + item, tile_amax);
          }
        }
      } else if constexpr (EPI == EPI_POWER) {
        // cosine part in columns [0, BN/2), sine part of the same bins in [BN/2, BN); warp cg owns 32 bins
        float re[32], im[32];
        tmem_ld32(t_row + cg * 32, re);
        tmem_ld32(t_row + BN / 2 + cg * 32, im);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        const long long rowi_c = static_cast<long long>(b) * 2 * p.M + m;
        if (row_ok && in_bounds(p.err, (rowi_c + p.M) * p.pw_ld + nt * (BN / 2) + cg * 32, 32, p.pw_elems,
                                SITE_GEMM_POWER)) {
          const int bin0 = nt * (BN / 2) + cg * 32;
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
      } else {  // EPI_MEL: warp cg owns 32 mel bins
        float v[32];
        tmem_ld32(t_row + cg * 32, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        const int n0 = nt * BN + cg * 32;
        float local_max = 0.0f;
        const int n_hi = (p.n_valid - n0 < 32 ? p.n_valid - n0 : 32) - 1;   // last bin this warp writes
        if (row_ok && n0 < p.n_valid &&
            in_bounds(p.err, (static_cast<long long>(b) * p.n_valid + n0 + n_hi) * p.M + m, 1, p.mel_elems,
                      SITE_GEMM_MEL)) {
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
        if (lane == 0 && local_max > 0.0f && in_bounds(p.err, b, 1, p.batch, SITE_GEMM_MEL))
          atomic_max_nonneg(p.mel_max + b, local_max);
      }
    }

    if (lane == 0) bulk_wait0();   // stores complete before the CTA (and its smem) goes away
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace wb
