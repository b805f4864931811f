// Fused non-causal self-attention for the encoder (head dim 64), sm_103a.
//
// The whisper-blaze showcase site, "The Solution" (flash_attn_hopper.cu card)
// and "Impact" ("Attention without the quadratic write"): online softmax over
// key tiles, scores never written to HBM.  Here rebuilt on tcgen05:
//   S_j = Q K_j^T      -> TMEM (two 128-column buffers, fp32)
//   P_j = exp(S_j - m) -> bf16 in shared memory (128-byte swizzled, K-major)
//   O_j = P_j V_j      -> TMEM (two 64-column buffers), folded into registers
//                         with the running rescale factor.
// One CTA owns 128 queries of one (batch, head).  Warp 0 lane 0 loads Q once
// and a ring of K / V^T tiles with TMA; warp 1 lane 0 issues the MMAs; warps
// 2-5 own one query row per thread (no cross-thread reductions).  Keys past
// the sequence end are masked to -inf; rows past it are not stored.
#pragma once
#include "ptx.cuh"
#include "types.h"

namespace wb {

// q / k maps: 3-D (d, T, batch) views of the query and key rows, box (64, 128, 1)
// vt map: 3-D (T, 64, batch*H) over V^T [batch*H][64][Tp], box (64, 64, 1)
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap vt_map, const __grid_constant__ AttnParams p) {
  using S = AttnSmem;
  constexpr uint32_t IDESC_S = make_idesc(128, ATT_BKV, 1u);
  constexpr uint32_t IDESC_O = make_idesc(128, ATT_HD, 1u);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base_u32 - smem_u32(smem_raw));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;                  // [STAGES]
  uint64_t* kv_empty = kv_full + ATT_STAGES;     // [STAGES]
  uint64_t* s_full = kv_empty + ATT_STAGES;      // [2]
  uint64_t* p_full = s_full + 2;                 // [2]
  uint64_t* o_full = p_full + 2;                 // [2]
  uint64_t* o_empty = o_full + 2;                // [2]
  uint64_t* mma_done = o_empty + 2;
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
    for (int s = 0; s < ATT_STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 128);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S buffers at 0 and 128, O tiles at 256 and 320.

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&q_map);
      tma_prefetch_desc(&k_map);
      tma_prefetch_desc(&vt_map);
      mbar_arrive_expect_tx(q_full, S::Q_BYTES);
      tma_load_3d(smem + S::OFF_Q, &q_map, q_full, h * ATT_HD, q0, b);
      uint32_t issued = 0, last_par = 0;
      bool ok = true;
      for (int j = 0; j < nkv && ok; ++j) {
        const int st = j % ATT_STAGES;
        const uint32_t ph = (j / ATT_STAGES) & 1;
        if (!mbar_wait(&kv_empty[st], ph ^ 1u, p.err, abort_flag, 11)) { ok = false; break; }
        mbar_arrive_expect_tx(&kv_full[st], S::K_BYTES + S::V_BYTES);
        const int kv0 = j * ATT_BKV;
        tma_load_3d(smem + S::OFF_K + st * S::K_BYTES, &k_map, &kv_full[st], h * ATT_HD, kv0, b);
        uint8_t* vdst = smem + S::OFF_V + st * S::V_BYTES;
        tma_load_3d(vdst, &vt_map, &kv_full[st], kv0, 0, bh);
        tma_load_3d(vdst + ATT_HD * 128, &vt_map, &kv_full[st], kv0 + 64, 0, bh);
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
      const uint32_t sq = smem_u32(smem + S::OFF_Q);
      bool ok = mbar_wait(q_full, 0, p.err, abort_flag, 12);
      auto issue_qk = [&](int j) -> bool {
        const int st = j % ATT_STAGES;
        if (!mbar_wait(&kv_full[st], (j / ATT_STAGES) & 1, p.err, abort_flag, 13)) return false;
        tc_fence_after();
        const uint32_t sk = smem_u32(smem + S::OFF_K + st * S::K_BYTES);
        const uint32_t d_tm = tmem + (j & 1) * ATT_BKV;
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_bf16(d_tm, sw128_desc(sq + k * 32), sw128_desc(sk + k * 32), IDESC_S, k != 0);
        mma_commit(&s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && nkv > 1) ok = issue_qk(1);
      for (int j = 0; j < nkv && ok; ++j) {
        const int st = j % ATT_STAGES;
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, p.err, abort_flag, 14)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(&o_empty[j & 1], ((j - 2) >> 1) & 1, p.err, abort_flag, 15)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sp = smem_u32(smem + S::OFF_P + (j & 1) * S::P_BYTES);
        const uint32_t sv = smem_u32(smem + S::OFF_V + st * S::V_BYTES);
        const uint32_t o_tm = tmem + 256 + (j & 1) * ATT_HD;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t half = (k >> 2) * (ATT_BQ * 128), off = (k & 3) * 32;
          const uint32_t vhalf = (k >> 2) * (ATT_HD * 128);
          mma_bf16(o_tm, sw128_desc(sp + half + off), sw128_desc(sv + vhalf + off), IDESC_O, k != 0);
        }
        mma_commit(&o_full[j & 1]);
        mma_commit(&kv_empty[st]);
        if (j + 2 < nkv) ok = issue_qk(j + 2);
      }
      mma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // --------------------------- softmax / output --------------------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float o_acc[ATT_HD];
#pragma unroll
    for (int e = 0; e < ATT_HD; ++e) o_acc[e] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;
    float alpha_q[2] = {1.0f, 1.0f};
    bool ok = true;

    auto consume_o = [&](int j) -> bool {
      if (!mbar_wait(&o_full[j & 1], (j >> 1) & 1, p.err, abort_flag, 16)) return false;
      tc_fence_after();
      const float a = alpha_q[j & 1];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_off + 256 + (j & 1) * ATT_HD + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o_acc[c * 32 + i] = o_acc[c * 32 + i] * a + v[i];
      }
      tc_fence_before();
      mbar_arrive(&o_empty[j & 1]);
      return true;
    };

    for (int j = 0; j < nkv && ok; ++j) {
      if (j >= 2 && !(ok = consume_o(j - 2))) break;
      if (!mbar_wait(&s_full[j & 1], (j >> 1) & 1, p.err, abort_flag, 17)) { ok = false; break; }
      tc_fence_after();
      float s[ATT_BKV];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_off + (j & 1) * ATT_BKV + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = v[i];
      }
      tmem_ld_wait();
      const int valid = min(ATT_BKV, p.T - j * ATT_BKV);
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < ATT_BKV; ++i) {
        s[i] = (i < valid) ? s[i] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[i]);
      }
      const float m_new = fmaxf(m_run, mx);
      const float alpha = ex2_approx(m_run - m_new);
      alpha_q[j & 1] = alpha;
      m_run = m_new;
      float sum = 0.0f;
      uint8_t* pbuf = smem + S::OFF_P + (j & 1) * S::P_BYTES;
#pragma unroll
      for (int c8 = 0; c8 < ATT_BKV / 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float p0 = ex2_approx(s[c8 * 8 + 2 * i] - m_new);
          const float p1 = ex2_approx(s[c8 * 8 + 2 * i + 1] - m_new);
          sum += p0 + p1;
          w[i] = pack_bf16(p0, p1);
        }
        const int half = c8 >> 3, chunk = c8 & 7;
        uint8_t* dst = pbuf + half * (ATT_BQ * 128) + r * 128 + ((chunk ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run = l_run * alpha + sum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }
    if (ok && nkv >= 2) ok = consume_o(nkv - 2);
    if (ok) ok = consume_o(nkv - 1);
    if (ok) {
      const int q = q0 + r;
      if (q < p.T) {
        const float inv = 1.0f / l_run;
        uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<long long>(b) * p.T + q) * p.d + h * ATT_HD);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          dst[j] = make_uint4(pack_bf16(o_acc[8 * j + 0] * inv, o_acc[8 * j + 1] * inv),
                              pack_bf16(o_acc[8 * j + 2] * inv, o_acc[8 * j + 3] * inv),
                              pack_bf16(o_acc[8 * j + 4] * inv, o_acc[8 * j + 5] * inv),
                              pack_bf16(o_acc[8 * j + 6] * inv, o_acc[8 * j + 7] * inv));
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
