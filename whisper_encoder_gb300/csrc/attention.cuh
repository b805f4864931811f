// Fused non-causal self-attention for the encoder (head dim 64), sm_103a.
//
// The whisper-blaze showcase site, "The Solution" (flash_attn_hopper.cu card)
// and "Impact" ("Attention without the quadratic write"): online softmax over
// key tiles, scores never written to HBM.  Rebuilt on tcgen05:
//   S_t = Q_t K_j^T        -> TMEM, fp32, one 128-column buffer per query tile
//   P_t = 2^(S_t c - m_t)  -> f16, written back over S_t in TMEM (packed ex2: two
//                             exponentials per MUFU op); the PV MMA reads its A operand from TMEM
//   O_t += P_t [V_j | 1]   -> TMEM, fp32, 80 columns: 64 of output and 16 copies of the
//                             row sum (a block of ones appended to V^T in shared memory)
// A CTA owns two 128-query tiles of one (batch, head).  Warp 0 lane 0 loads
// both Q tiles once and a ring of K / V^T tiles with TMA; warp 1 lane 0 issues
// the MMAs, alternating between the tiles so that one tile's matrix products
// run while the other tile's softmax runs; warps 2-17 split each query row of
// the two tiles over two threads (64 score columns each).  The running max m_t is only moved
// (and O rescaled in TMEM) when a new row maximum exceeds it by more than a
// factor 2^8, which keeps every P entry below 256.  Keys past the sequence
// end are masked to -inf; rows past it are not stored.
#pragma once
#include "ptx.cuh"
#include "types.h"

namespace wb {

// q / k maps: 3-D (d, T, batch) views of the query and key rows (bf16), box (64, 128, 1)
// vt map: 3-D (T, 64, batch*H) over V^T [batch*H][64][Tp] (f16), box (64, 64, 1)
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap vt_map, const __grid_constant__ AttnParams p) {
  using S = AttnSmem;
  constexpr uint32_t IDESC_S = make_idesc(128, ATT_BKV, 1u);    // bf16 x bf16
  constexpr uint32_t IDESC_O = make_idesc(128, ATT_NPV, 0u);    // f16 x f16
  constexpr float RESCALE_LOG2 = 8.0f;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_u32 - smem_u32(smem_raw));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;                  // [STAGES]
  uint64_t* kv_empty = kv_full + ATT_STAGES;     // [STAGES]
  uint64_t* s_full = kv_empty + ATT_STAGES;      // [TILES]
  uint64_t* p_full = s_full + ATT_TILES;         // [TILES]
  uint64_t* o_done = p_full + ATT_TILES;         // [TILES]
  uint64_t* xbar = o_done + ATT_TILES;           // [TILES][4]: row-max exchange between the two row halves
  uint64_t* mma_done = xbar + ATT_TILES * 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  const int n_qp = (p.T + ATT_TILES * ATT_BQ - 1) / (ATT_TILES * ATT_BQ);
  const int qp = blockIdx.x % n_qp;
  const int bh = blockIdx.x / n_qp;
  const int b = bh / p.H, h = bh % p.H;
  const int q0 = qp * ATT_TILES * ATT_BQ;
  const int nkv = (p.T + ATT_BKV - 1) / ATT_BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ATT_STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < ATT_TILES; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4 * ATT_HALVES);
      mbar_init(&o_done[t], 1);
      for (int q = 0; q < 4; ++q) mbar_init(&xbar[t * 4 + q], ATT_HALVES);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp >= 2) {
    // rows 64..79 of every V^T half tile hold f16 ones: their PV columns carry the row sums
    constexpr int ONES_CHUNKS = (ATT_NPV - ATT_HD) * 128 / 16;     // 16-byte chunks per half tile
    const int n16 = ATT_STAGES * 2 * ONES_CHUNKS;
    for (int i = threadIdx.x - 64; i < n16; i += ATT_THREADS - 64) {
      const int half = i / ONES_CHUNKS, within = i % ONES_CHUNKS;
      uint8_t* dst = smem + S::OFF_V + half * S::VH_BYTES + ATT_HD * 128 + within * 16;
      *reinterpret_cast<uint4*>(dst) = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S_t at 128 t, O_t at 256 + 128 t (80 columns each).

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&q_map);
      tma_prefetch_desc(&k_map);
      tma_prefetch_desc(&vt_map);
      mbar_arrive_expect_tx(q_full, ATT_TILES * S::Q_BYTES);
      for (int t = 0; t < ATT_TILES; ++t)
        tma_load_3d(smem + S::OFF_Q + t * S::Q_BYTES, &q_map, q_full, h * ATT_HD, q0 + t * ATT_BQ, b);
      uint32_t issued = 0, last_par = 0;
      bool ok = true;
      for (int j = 0; j < nkv && ok; ++j) {
        const int st = j % ATT_STAGES;
        const uint32_t ph = (j / ATT_STAGES) & 1;
        if (!mbar_wait(&kv_empty[st], ph ^ 1u, p.err, abort_flag, 11)) { ok = false; break; }
        mbar_arrive_expect_tx(&kv_full[st], S::K_BYTES + 2 * ATT_HD * 128);
        const int kv0 = j * ATT_BKV;
        tma_load_3d(smem + S::OFF_K + st * S::K_BYTES, &k_map, &kv_full[st], h * ATT_HD, kv0, b);
        uint8_t* vdst = smem + S::OFF_V + st * S::V_BYTES;
        tma_load_3d(vdst, &vt_map, &kv_full[st], kv0, 0, bh);
        tma_load_3d(vdst + S::VH_BYTES, &vt_map, &kv_full[st], kv0 + 64, 0, bh);
        issued |= 1u << st;
        last_par = (last_par & ~(1u << st)) | (ph << st);
      }
      if (!ok) {
        mbar_drain(q_full, 0);
        for (int s = 0; s < ATT_STAGES; ++s)
          if (issued & (1u << s)) mbar_drain(&kv_full[s], (last_par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // Descriptors are built once: for these shared-memory addresses (below 256 KB) the
      // descriptor of base + c is the descriptor of base plus c / 16, so every MMA only adds a
      // compile-time offset.  The K/V stage index advances incrementally (no division).
      const uint64_t q_desc0 = sw128_desc(smem_u32(smem + S::OFF_Q));
      const uint64_t k_desc0 = sw128_desc(smem_u32(smem + S::OFF_K));
      const uint64_t v_desc0 = sw128_desc(smem_u32(smem + S::OFF_V));
      auto pv = [&](int t, int vst, bool first) {
        // P_t sits in the first 64 columns of S_t (two f16 per column): 8 columns per K16 step
        const uint64_t vd = v_desc0 + static_cast<uint64_t>(vst * (S::V_BYTES >> 4));
        const uint32_t o_tm = tmem + 256 + t * 128;
        const uint32_t p_tm = tmem + t * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_tmem_a(o_tm, p_tm + k * 8, vd + (((k >> 2) * S::VH_BYTES + (k & 3) * 32) >> 4), IDESC_O,
                         (!first || k != 0) ? 1u : 0u);
        mma_commit(&o_done[t]);
      };
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag, 12);
      int st = 0, vst = 0;         // stage of K/V j, stage of V j-1
      uint32_t kv_phase = 0;
      for (int j = 0; j < nkv && ok; ++j) {
        if (!mbar_wait(&kv_full[st], kv_phase, p.err, abort_flag, 13)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kd = k_desc0 + static_cast<uint64_t>(st * (S::K_BYTES >> 4));
        for (int t = 0; t < ATT_TILES && ok; ++t) {
          if (j > 0) {
            if (!mbar_wait(&p_full[t], (j - 1) & 1, p.err, abort_flag, 14)) { ok = false; break; }
            tc_fence_after();
            pv(t, vst, j == 1);
          }
          const uint64_t qd = q_desc0 + static_cast<uint64_t>(t * (S::Q_BYTES >> 4));
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_bf16(tmem + t * 128, qd + 2 * k, kd + 2 * k, IDESC_S, k != 0);
          mma_commit(&s_full[t]);
        }
        if (ok && j > 0) mma_commit(&kv_empty[vst]);
        vst = st;
        if (++st == ATT_STAGES) { st = 0; kv_phase ^= 1u; }
      }
      for (int t = 0; t < ATT_TILES && ok; ++t) {
        if (!mbar_wait(&p_full[t], (nkv - 1) & 1, p.err, abort_flag, 15)) { ok = false; break; }
        tc_fence_after();
        pv(t, vst, nkv == 1);
      }
      mma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // --------------------------- softmax / output --------------------------
    // 16 warps: tile t = sw / 8, row half hf = (sw / 4) % 2 (score columns 64 hf .. 64 hf + 63),
    // TMEM lane quarter = warp % 4.  The two threads holding the halves of one row exchange
    // their half-row maxima through shared memory (one mbarrier per tile and lane quarter).
    const int sw = warp - 2;
    const int t = sw >> 3;
    const int hf = (sw >> 2) & 1;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + t * 128 + hf * 64;
    const uint32_t o_tm = tmem + lane_off + 256 + t * 128;
    const uint32_t p_tm = tmem + lane_off + t * 128 + hf * 32;   // this half's 32 packed P columns
    float* xmax = reinterpret_cast<float*>(smem + S::OFF_XMAX);
    uint64_t* xb = &xbar[t * 4 + quarter];
    const float c = p.scale_log2;
    float m_use = -INFINITY;
    bool ok = true;

    for (int j = 0; j < nkv && ok; ++j) {
      if (!mbar_wait(&s_full[t], j & 1, p.err, abort_flag, 16)) { ok = false; break; }
      tc_fence_after();
      float s[64];
      {
        float v[32];
        tmem_ld32(s_tm, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = v[i];
        tmem_ld32(s_tm + 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 + i] = v[i];
      }
      tmem_ld_wait();
      const int valid = p.T - j * ATT_BKV - hf * 64;      // columns of this half inside the sequence
      if (valid < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = (i < valid) ? s[i] : -INFINITY;
      }
      float m4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) m4[k] = fmaxf(s[2 * k], s[2 * k + 1]);       // s[0..7]
#pragma unroll
      for (int i = 8; i < 64; i += 8) {                                          // s[8..63], 8 per step
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmax3(m4[k], s[i + 2 * k], s[i + 2 * k + 1]);
      }
      const float own = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
      float* xm = xmax + ((j & 1) * ATT_TILES + t) * ATT_HALVES * ATT_BQ;
      xm[hf * ATT_BQ + r] = own;
      tc_fence_before();           // this half's TMEM loads of S precede the partner's P stores
      __syncwarp();
      if (lane == 0) mbar_arrive(xb);
      if (!mbar_wait(xb, j & 1, p.err, abort_flag, 19)) { ok = false; break; }
      tc_fence_after();
      const float mx = fmaxf(own, xm[(1 - hf) * ATT_BQ + r]);
      const float m_cand = mx * c;
      float alpha = 1.0f;
      bool rescale = false;
      if (j == 0) {
        m_use = m_cand;
      } else if (m_cand > m_use + RESCALE_LOG2) {
        alpha = ex2_approx(m_use - m_cand);
        m_use = m_cand;
        rescale = true;
      }
      if (j > 0) {
        // PV of the previous step is complete: P may be overwritten and O is stable until PV(j) is issued
        if (!mbar_wait(&o_done[t], (j - 1) & 1, p.err, abort_flag, 17)) { ok = false; break; }
        tc_fence_after();
      }
      const float mb = -m_use;
      uint32_t pw[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) pw[i] = ex2_f16x2(pack_f16(fmaf(s[2 * i], c, mb), fmaf(s[2 * i + 1], c, mb)));
      // Half 1's P columns (32..63) overlay half 0's scores; half 0 finished reading them before
      // it arrived at the row-max exchange, which half 1 has passed.
      tmem_st32u(p_tm, pw);
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // half 0 rescales O columns 0..31 and the row sums 64..79, half 1 columns 32..63
        float v[32];
        tmem_ld32(o_tm + hf * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= alpha;
        tmem_st32(o_tm + hf * 32, v);
        if (hf == 0) {
          float w[16];
          tmem_ld16(o_tm + 64, w);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] *= alpha;
          tmem_st16(o_tm + 64, w);
        }
        tmem_st_wait();
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    if (ok && mbar_wait(&o_done[t], (nkv - 1) & 1, p.err, abort_flag, 18)) {
      tc_fence_after();
      float o[32], w[16];
      tmem_ld32(o_tm + hf * 32, o);
      tmem_ld16(o_tm + 64, w);
      tmem_ld_wait();
      const int q = q0 + t * ATT_BQ + r;
      if (q < p.T) {
        const float inv = 1.0f / w[0];
        uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<long long>(b) * p.T + q) * p.d + h * ATT_HD + hf * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          dst[k] = make_uint4(pack_bf16(o[8 * k + 0] * inv, o[8 * k + 1] * inv),
                              pack_bf16(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                              pack_bf16(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                              pack_bf16(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace wb
