// Fused non-causal self-attention for the encoder (head dim 64), sm_103a.
//
// The whisper-blaze showcase site, "The Solution" (flash_attn_hopper.cu card)
// and "Impact" ("Attention without the quadratic write"): online softmax over
// key tiles, scores never written to HBM.  Rebuilt on tcgen05:
//   S = Q K_j^T          -> TMEM, fp32, 128 columns
//   P = 2^(S c - m)      -> f16 in TMEM, 64 columns (packed ex2: two exponentials per MUFU op);
//                           the PV MMA reads its A operand from TMEM
//   l += rowsum(P)       -> registers (packed f16 adds within a key tile, fp32 across tiles)
//   O += P V_j           -> TMEM, fp32, 64 columns
// A CTA owns one 128-query tile of one (batch, head) and 256 TMEM columns, so
// two CTAs share an SM: one CTA's prologue (Q and first K/V loads) and epilogue
// run under the other's main loop, and each has its own MMA issuer.  Warp 0
// lane 0 loads Q once and rings of K and V^T tiles with TMA; warp 1 lane 0
// issues the MMAs; warps 2-9 run the softmax, each row held by four threads of
// one warp (32 score columns each).  A softmax thread releases S as soon as it has loaded it into
// registers, so QK of key tile j+1 runs while the softmax of key tile j is
// still exponentiating; the softmax only waits for PV of key tile j-1 before
// it overwrites P.  The running max m is only moved (and O rescaled in TMEM)
// when a new row maximum exceeds it by more than a factor 2^8, which keeps
// every P entry below 256.  Keys past the sequence end are masked to -inf;
// rows past it are not stored.
#pragma once
#include "ptx.cuh"
#include "types.h"

namespace wb {

// q / k maps: 3-D (d, T, batch) views of the query and key rows (bf16), box (64, 128, 1)
// vt map: 3-D (T, 64, batch*H) over V^T [batch*H][64][Tp] (f16), box (64, 64, 1)
__global__ void __launch_bounds__(ATT_THREADS, ATT_CTAS_PER_SM)
    attention_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap vt_map, const __grid_constant__ AttnParams p) {
  using S = AttnSmem;
  constexpr uint32_t IDESC_S = make_idesc(128, ATT_BKV, 1u);    // bf16 x bf16
  constexpr uint32_t IDESC_O = make_idesc(128, ATT_HD, 0u);     // f16 x f16
  constexpr float RESCALE_LOG2 = 8.0f;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_u32 - smem_u32(smem_raw));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;                 // [KSTAGES]
  uint64_t* k_empty = k_full + ATT_KSTAGES;      // [KSTAGES]
  uint64_t* v_full = k_empty + ATT_KSTAGES;      // [VSTAGES]
  uint64_t* v_empty = v_full + ATT_VSTAGES;      // [VSTAGES]
  uint64_t* s_full = v_empty + ATT_VSTAGES;      // QK done: S holds the scores
  uint64_t* s_free = s_full + 1;                 // S loaded by all softmax warps
  uint64_t* p_full = s_free + 1;                 // P written
  uint64_t* pv_done = p_full + 1;                // PV done: P free, O stable
  uint64_t* mma_done = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  const int n_qt = (p.T + ATT_BQ - 1) / ATT_BQ;
  const int qt = blockIdx.x % n_qt;
  const int bh = blockIdx.x / n_qt;
  const int b = bh / p.H, h = bh % p.H;
  const int q0 = qt * ATT_BQ;
  const int nkv = (p.T + ATT_BKV - 1) / ATT_BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ATT_KSTAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < ATT_VSTAGES; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, ATT_SOFTMAX_WARPS);
    mbar_init(p_full, ATT_SOFTMAX_WARPS);
    mbar_init(pv_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, ATT_TM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // barriers and TMEM are set up: from here on the kernel reads its inputs
  grid_dependency_wait();
  grid_dependents_launch();

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&q_map);
      tma_prefetch_desc(&k_map);
      tma_prefetch_desc(&vt_map);
      mbar_arrive_expect_tx(q_full, S::Q_BYTES);
      tma_load_3d(smem + S::OFF_Q, &q_map, q_full, h * ATT_HD, q0, b);
      // Load order K_0, then (K_{i+1}, V_i): the MMA warp consumes K one key tile ahead of V.
      uint32_t k_issued = 0, k_par = 0, v_issued = 0, v_par = 0;
      auto load_k = [&](int jj) -> bool {
        const int st = jj % ATT_KSTAGES;
        const uint32_t ph = (jj / ATT_KSTAGES) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1u, p.err, abort_flag, 11)) return false;
        mbar_arrive_expect_tx(&k_full[st], S::K_BYTES);
        tma_load_3d(smem + S::OFF_K + st * S::K_BYTES, &k_map, &k_full[st], h * ATT_HD, jj * ATT_BKV, b);
        k_issued |= 1u << st;
        k_par = (k_par & ~(1u << st)) | (ph << st);
        return true;
      };
      auto load_v = [&](int jj) -> bool {
        const int st = jj % ATT_VSTAGES;
        const uint32_t ph = (jj / ATT_VSTAGES) & 1;
        if (!mbar_wait(&v_empty[st], ph ^ 1u, p.err, abort_flag, 10)) return false;
        mbar_arrive_expect_tx(&v_full[st], S::V_BYTES);
        uint8_t* vdst = smem + S::OFF_V + st * S::V_BYTES;
        tma_load_3d(vdst, &vt_map, &v_full[st], jj * ATT_BKV, 0, bh);
        tma_load_3d(vdst + S::VH_BYTES, &vt_map, &v_full[st], jj * ATT_BKV + 64, 0, bh);
        v_issued |= 1u << st;
        v_par = (v_par & ~(1u << st)) | (ph << st);
        return true;
      };
      bool ok = load_k(0);
      for (int i = 0; i < nkv && ok; ++i) {
        if (i + 1 < nkv) ok = load_k(i + 1);
        ok = ok && load_v(i);
      }
      if (!ok) {
        // copies already issued still land in shared memory: wait for them before the CTA exits
        mbar_drain(q_full, 0);
        for (int s = 0; s < ATT_KSTAGES; ++s)
          if (k_issued & (1u << s)) mbar_drain(&k_full[s], (k_par >> s) & 1u);
        for (int s = 0; s < ATT_VSTAGES; ++s)
          if (v_issued & (1u << s)) mbar_drain(&v_full[s], (v_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // For these shared-memory addresses (below 256 KB) the descriptor of base + c is the
      // descriptor of base plus c / 16, so every MMA only adds an offset.
      const uint64_t q_desc = sw128_desc(smem_u32(smem + S::OFF_Q));
      const uint64_t k_desc0 = sw128_desc(smem_u32(smem + S::OFF_K));
      const uint64_t v_desc0 = sw128_desc(smem_u32(smem + S::OFF_V));
      auto qk = [&](int jj) -> bool {
        // S = Q K_jj^T once K_jj has landed and the softmax has loaded S of key tile jj - 1
        const int st = jj % ATT_KSTAGES;
        if (!mbar_wait(&k_full[st], (jj / ATT_KSTAGES) & 1, p.err, abort_flag, 13)) return false;
        if (jj > 0 && !mbar_wait(s_free, (jj - 1) & 1, p.err, abort_flag, 20)) return false;
        tc_fence_after();
        const uint64_t kd = k_desc0 + static_cast<uint64_t>(st * (S::K_BYTES >> 4));
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_bf16(tmem + ATT_TM_S, q_desc + 2 * k, kd + 2 * k, IDESC_S, k != 0);
        mma_commit(s_full);
        mma_commit(&k_empty[st]);
        return true;
      };
      auto pv = [&](int jj) -> bool {
        // O += P V_jj; P holds 128 keys as 64 packed f16 columns: 8 columns per K16 step
        const int st = jj % ATT_VSTAGES;
        if (!mbar_wait(&v_full[st], (jj / ATT_VSTAGES) & 1, p.err, abort_flag, 21)) return false;
        if (!mbar_wait(p_full, jj & 1, p.err, abort_flag, 14)) return false;
        tc_fence_after();
        const uint64_t vd = v_desc0 + static_cast<uint64_t>(st * (S::V_BYTES >> 4));
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_tmem_a(tmem + ATT_TM_O, tmem + ATT_TM_P + k * 8,
                         vd + (((k >> 2) * S::VH_BYTES + (k & 3) * 32) >> 4), IDESC_O,
                         (jj > 0 || k != 0) ? 1u : 0u);
        mma_commit(pv_done);
        mma_commit(&v_empty[st]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag, 12) && qk(0);
      for (int j = 0; j < nkv && ok; ++j) {
        if (j + 1 < nkv) ok = qk(j + 1);
        ok = ok && pv(j);
      }
      mma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // --------------------------- softmax / output --------------------------
    // 8 warps; warp w owns the 16 TMEM lanes (query rows) 32 (w % 4) + 16 sub .. + 15, sub = (w - 2) / 4.
    // With the 16-lane TMEM shapes thread t holds rows ra = t/4 and ra + 8 of that block and, of each,
    // the score columns 8k + 2 (t % 4) and + 1 (k = 0..15): 32 of the row's 128 scores.  The four
    // threads that share a row combine row maxima with two shuffles and keep partial row sums.  A
    // thread's pair of adjacent scores becomes one packed f16 P column, 4k + t % 4, which is where the
    // 16x128b store shape puts it.  Waits are made warp-uniform so that a timeout leaves no lane behind.
    const int quarter = warp & 3;
    const int sub = ((warp - 2) >> 2) & 1;
    const int lane_base = quarter * 32 + sub * 16;
    const uint32_t lane_off = static_cast<uint32_t>(lane_base) << 16;
    const uint32_t s_tm = tmem + lane_off + ATT_TM_S;
    const uint32_t o_tm = tmem + lane_off + ATT_TM_O;
    const uint32_t p_tm = tmem + lane_off + ATT_TM_P;
    const int ra = lane_base + (lane >> 2);        // first of this thread's two rows inside the tile
    const int cq = 2 * (lane & 3);                 // this thread's column offset in every 8-column group
    const float c = p.scale_log2;
    float m_a = -INFINITY, m_b = -INFINITY;        // running maxima (log2 units) of rows ra and ra + 8
    float l_a = 0.0f, l_b = 0.0f;                  // this thread's share of the two row sums, scaled like O
    bool ok = true;

    for (int j = 0; j < nkv && ok; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(s_full, j & 1, p.err, abort_flag, 16))) { ok = false; break; }
      tc_fence_after();
      // s[4k], s[4k+1]: row ra, columns 8k + cq, + 1; s[4k+2], s[4k+3]: row ra + 8, same columns
      float s[64];
      {
        uint32_t v[32];
        tmem_ld_16x256b_x8(s_tm, v);               // columns 0..63
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(v[i]);
        tmem_ld_16x256b_x8(s_tm + 64, v);          // columns 64..127
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 + i] = __uint_as_float(v[i]);
      }
      tmem_ld_wait();
      tc_fence_before();           // S is in registers: QK of the next key tile may overwrite it
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      const int valid = p.T - j * ATT_BKV;         // key columns of this tile inside the sequence
      if (valid < ATT_BKV) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const int col = 8 * kk + cq;
          if (col >= valid) s[4 * kk] = s[4 * kk + 2] = -INFINITY;
          if (col + 1 >= valid) s[4 * kk + 1] = s[4 * kk + 3] = -INFINITY;
        }
      }
      // this thread's share (32 scores) of the maxima of rows ra and ra + 8
      float xa0 = fmaxf(s[0], s[1]), xa1 = fmaxf(s[4], s[5]);
      float xb0 = fmaxf(s[2], s[3]), xb1 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int kk = 2; kk < 16; kk += 2) {
        xa0 = fmax3(xa0, s[4 * kk], s[4 * kk + 1]);
        xa1 = fmax3(xa1, s[4 * kk + 4], s[4 * kk + 5]);
        xb0 = fmax3(xb0, s[4 * kk + 2], s[4 * kk + 3]);
        xb1 = fmax3(xb1, s[4 * kk + 6], s[4 * kk + 7]);
      }
      float xa = fmaxf(xa0, xa1), xb = fmaxf(xb0, xb1);
      float alpha_a = 1.0f, alpha_b = 1.0f;
      bool rescale = false;
      // From the second key tile on, the running maxima only move where a row's new maximum passes
      // them by more than 2^8; a vote on the threads' partial maxima finds the (rare) tiles where that
      // can happen, and only those pay for combining the row maxima across the four threads of a row.
      if (j == 0 || __any_sync(0xffffffffu, xa * c > m_a + RESCALE_LOG2 || xb * c > m_b + RESCALE_LOG2)) {
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 1));
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 2));
        const float ca = xa * c, cb = xb * c;
        if (j == 0) {
          m_a = ca;
          m_b = cb;
        } else {
          if (ca > m_a + RESCALE_LOG2) {
            alpha_a = ex2_approx(m_a - ca);
            m_a = ca;
            l_a *= alpha_a;
            rescale = true;
          }
          if (cb > m_b + RESCALE_LOG2) {
            alpha_b = ex2_approx(m_b - cb);
            m_b = cb;
            l_b *= alpha_b;
            rescale = true;
          }
        }
      }
      // pw[2k]: row ra, P column 4k + t % 4 (keys 8k + cq, + 1); pw[2k+1]: row ra + 8, same column
      const uint64_t c2 = f32x2_pack(c, c), na2 = f32x2_pack(-m_a, -m_a), nb2 = f32x2_pack(-m_b, -m_b);
      uint32_t pw[32];
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        float x0, x1, x2, x3;
        fma_f32x2(x0, x1, s[4 * kk], s[4 * kk + 1], c2, na2);
        fma_f32x2(x2, x3, s[4 * kk + 2], s[4 * kk + 3], c2, nb2);
        pw[2 * kk] = ex2_f16x2(pack_f16(x0, x1));
        pw[2 * kk + 1] = ex2_f16x2(pack_f16(x2, x3));
      }
      {
        // partial row sums of the 32 f16 entries per row: pairwise packed adds (partial sums stay
        // below 2^12), then fp32
        uint32_t a[8], bq[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          a[i] = hadd2_u32(pw[4 * i], pw[4 * i + 2]);
          bq[i] = hadd2_u32(pw[4 * i + 1], pw[4 * i + 3]);
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1) {
#pragma unroll
          for (int i = 0; i < w; ++i) {
            a[i] = hadd2_u32(a[i], a[i + w]);
            bq[i] = hadd2_u32(bq[i], bq[i + w]);
          }
        }
        l_a += f16x2_sum_f32(a[0]);
        l_b += f16x2_sum_f32(bq[0]);
      }
      // PV of key tile j-1 is done: P may be overwritten and O is stable until PV of tile j is issued
      if (j > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, p.err, abort_flag, 17))) { ok = false; break; }
        tc_fence_after();
      }
      tmem_st_16x128b_x16(p_tm, pw);
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        uint32_t v[32];
        tmem_ld_16x256b_x8(o_tm, v);
        tmem_ld_wait();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          v[4 * kk] = __float_as_uint(__uint_as_float(v[4 * kk]) * alpha_a);
          v[4 * kk + 1] = __float_as_uint(__uint_as_float(v[4 * kk + 1]) * alpha_a);
          v[4 * kk + 2] = __float_as_uint(__uint_as_float(v[4 * kk + 2]) * alpha_b);
          v[4 * kk + 3] = __float_as_uint(__uint_as_float(v[4 * kk + 3]) * alpha_b);
        }
        tmem_st_16x256b_x8(o_tm, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // full row sums from the four threads of each row
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    if (ok && __all_sync(0xffffffffu, mbar_wait(pv_done, (nkv - 1) & 1, p.err, abort_flag, 18))) {
      tc_fence_after();
      uint32_t v[32];                              // [4k..4k+3]: rows ra / ra + 8, columns 8k + cq, + 1
      tmem_ld_16x256b_x8(o_tm, v);
      tmem_ld_wait();
      const float ia = 1.0f / l_a, ib = 1.0f / l_b;
      const int qa = q0 + ra, qb = qa + 8;
      __nv_bfloat16* oa = p.out + (static_cast<long long>(b) * p.T + qa) * p.d + h * ATT_HD + cq;
      __nv_bfloat16* ob = oa + 8LL * p.d;
      uint32_t mx2 = 0u;                           // packed |bf16| maxima of the stored outputs
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t wa = pack_bf16(__uint_as_float(v[4 * kk]) * ia, __uint_as_float(v[4 * kk + 1]) * ia);
        const uint32_t wb = pack_bf16(__uint_as_float(v[4 * kk + 2]) * ib, __uint_as_float(v[4 * kk + 3]) * ib);
        const long long out_el = static_cast<long long>(p.batch) * p.T * p.d;
        if (qa < p.T && in_bounds(p.err, (oa + 8 * kk) - p.out, 2, out_el, SITE_ATT_OUT)) {
          *reinterpret_cast<uint32_t*>(oa + 8 * kk) = wa;
          mx2 = bf16x2_max(mx2, wa & 0x7fff7fffu);
        }
        if (qb < p.T && in_bounds(p.err, (ob + 8 * kk) - p.out, 2, out_el, SITE_ATT_OUT)) {
          *reinterpret_cast<uint32_t*>(ob + 8 * kk) = wb;
          mx2 = bf16x2_max(mx2, wb & 0x7fff7fffu);
        }
      }
      if (p.amax) {   // one atomic per warp: the per-chunk scale of an E4M3 out-projection operand
        float mx = fmaxf(__uint_as_float(mx2 << 16), __uint_as_float(mx2 & 0xffff0000u));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0 && mx > 0.0f && in_bounds(p.err, b, 1, p.batch, SITE_ATT_AMAX)) atomic_max_nonneg(p.amax + b, mx);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, ATT_TM_COLS);
}

}  // namespace wb
