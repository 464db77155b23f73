// decode_kernel.cuh -- split-KV partials of the multi-token (MTP-verify) decode.
//
// The MiMo-V2-Flash Technical Report (§2.3.1) verifies 1 + K draft tokens in
// one pass over the KV cache; this kernel computes, for one chunk of the cache
// of one (sequence, KV head) at a time, the unnormalised attention partials of
// eqs. (1)-(3) of §2.2 for the T new tokens x G query heads of that KV head:
// the running max m, the sum l of 2^(a - m) and O = sum 2^(a - m) v, without
// the sink (sinkattn_combine_kernel adds it once, over all chunks).
//
// The cache is streamed in 64-key blocks, four in flight (TMA into a shared
// memory ring); S = Q K^T and O += P V run on tcgen05 with S, P and O in TMEM.
// Only the T * G <= 128 packed rows that exist are touched by the softmax.
//
// Warp roles (384 threads, one CTA per SM):
//   warp 0       TMA producer: Q tile once per chunk, K/V blocks.
//   warp 1       MMA issuer: S = Q K^T (12 k-steps), then O += P V.
//   warp 2       TMEM allocator (S0, S1, O: 256 columns).
//   warps 4-7    online softmax, one row per thread: the block's masked max
//                (3-input max), lazy running max (moves only when a block
//                exceeds it by more than 2^8), P = 2^(s * scale * log2e - m) as
//                bf16 pairs into TMEM, l, and the rescale of this row's O when
//                m moves; at the end of a chunk the partial row is written.
//   warps 8-11   RoPE on dims 0..63 of the Q tile and of every K block.
#pragma once
#include "attn_kernel.cuh"
#include "common.cuh"

namespace sa {

constexpr int32_t kDecBN = 64;      // keys per block
constexpr int32_t kDecStages = 4;   // K/V blocks in flight
constexpr uint32_t kDecTmemCols = 256;
constexpr uint32_t kDecTmemO = 128;

struct DecLayout {
  static constexpr uint32_t kKBox = kDecBN * kRowBytes;    // 64 keys x 64 dims: 8 KB
  static constexpr uint32_t kQOff = 0;                     // 128 rows x 3 boxes: 48 KB
  static constexpr uint32_t kKVOff = kQStageBytes;
  static constexpr uint32_t kKVStage = 5 * kKBox;          // K: 3 boxes, V: 2 boxes
  static constexpr uint32_t kBarOff = kKVOff + kDecStages * kKVStage;
  // q_full q_ready q_empty | kv_full[S] k_ready[S] kv_empty[S] | s_full[2] p_full[2] pv_done o_empty drain
  static constexpr uint32_t kNumBars = 3 + 3 * kDecStages + 7;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;  // tmem slot, abort flag
  static constexpr uint32_t kTurnsOff = (kMiscOff + 16 + 7) & ~7u;
  static constexpr uint32_t kBytes = kTurnsOff + 32 * 8;
  static constexpr uint32_t kDynSmem = kBytes + 1024;
};
static_assert(DecLayout::kDynSmem <= 232448, "decode kernel shared memory");

__global__ void __launch_bounds__(kThreads, 1)
    sinkattn_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ AttnArgs args) {
  using Ly = DecLayout;
  constexpr int32_t S = kDecStages;
  constexpr int32_t BN = kDecBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int32_t warp = threadIdx.x >> 5;
  const int32_t lane = threadIdx.x & 31;

  auto bar = [&](uint32_t i) { return sbase + Ly::kBarOff + i * 8; };
  const uint32_t B_QFULL = bar(0), B_QREADY = bar(1), B_QEMPTY = bar(2);
  auto B_KVFULL = [&](uint32_t s) { return bar(3 + s); };
  auto B_KREADY = [&](uint32_t s) { return bar(3 + S + s); };
  auto B_KVEMPTY = [&](uint32_t s) { return bar(3 + 2 * S + s); };
  auto B_SFULL = [&](uint32_t b) { return bar(3 + 3 * S + b); };
  auto B_PFULL = [&](uint32_t b) { return bar(3 + 3 * S + 2 + b); };
  const uint32_t B_PVDONE = bar(3 + 3 * S + 4);
  const uint32_t B_OEMPTY = bar(3 + 3 * S + 5);
  const uint32_t B_DRAIN = bar(3 + 3 * S + 6);

  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  unsigned long long *turns = reinterpret_cast<unsigned long long *>(smem + Ly::kTurnsOff);

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    mbar_init(B_QFULL, 1);
    mbar_init(B_QREADY, 128);
    mbar_init(B_QEMPTY, 1);
    for (uint32_t s = 0; s < S; ++s) {
      mbar_init(B_KVFULL(s), 1);
      mbar_init(B_KREADY(s), 128);
      mbar_init(B_KVEMPTY(s), 1);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(B_SFULL(b), 1);
      mbar_init(B_PFULL(b), 128);
    }
    mbar_init(B_PVDONE, 1);
    mbar_init(B_OEMPTY, 128);
    mbar_init(B_DRAIN, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) turns[threadIdx.x] = args.rope_turns[threadIdx.x];
  if (warp == 2) {
    tmem_alloc(sbase + Ly::kMiscOff, kDecTmemCols);
    tmem_relinquish();
  }
  // The Q tile has T * G rows; the MMA reads all 128, so the rest stay zero.
  for (uint32_t i = threadIdx.x; i < kQStageBytes / 16; i += kThreads)
    reinterpret_cast<uint4 *>(smem + Ly::kQOff)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int32_t G = args.G;
  const int32_t R = args.part_rows;  // T * G packed rows

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t gq = 0, gk = 0;
      bool ok = true;
      for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
        const Item it = make_item(args, w, BN);
        if (!it.valid) continue;
        if (!(ok = wait_bar(B_QEMPTY, (gq & 1) ^ 1, abort_flag, 1))) break;
        mbar_arrive_expect_tx(B_QFULL, args.q_tx_bytes);
#pragma unroll
        for (int c = 0; c < 3; ++c)
          tma_load_3d(sbase + Ly::kQOff + c * kQBoxBytes, &tm_q, c * 64, it.kvh * G, it.q_row, B_QFULL);
        ++gq;
        for (int32_t j = 0; j < it.n_blk; ++j) {
          const uint32_t st = gk % S;
          if (!(ok = wait_bar(B_KVEMPTY(st), ((gk / S) & 1) ^ 1, abort_flag, 2))) break;
          mbar_arrive_expect_tx(B_KVFULL(st), Ly::kKVStage);
          const uint32_t dst = sbase + Ly::kKVOff + st * Ly::kKVStage;
          const int32_t krow = it.kv_row0 + it.kstart + j * BN;
#pragma unroll
          for (int c = 0; c < 3; ++c)
            tma_load_3d(dst + c * Ly::kKBox, &tm_k, c * 64, it.kvh, krow, B_KVFULL(st));
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_3d(dst + (3 + c) * Ly::kKBox, &tm_v, c * 64, it.kvh, krow, B_KVFULL(st));
          ++gk;
        }
      }
      if (gq > 0) drain_wait(B_QFULL, (gq - 1) & 1);
      for (uint32_t s = 0; s < S; ++s)
        if (gk > s) drain_wait(B_KVFULL(s), ((gk - 1 - s) / S) & 1);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t rot = args.rope_on ? 0u : 1u;  // rotated dims are fp16
      const uint32_t kIdQK = idesc_f32acc(128, BN, 1, 0, 0);
      const uint32_t kIdQKRot = idesc_f32acc(128, BN, rot, 0, 0);
      constexpr uint32_t kIdPV = idesc_f32acc(128, kDv, 1, 0, 1);
      constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
      const uint32_t q_lo = ((sbase + Ly::kQOff) >> 4) | (1u << 16);
      const uint32_t kv_lo = ((sbase + Ly::kKVOff) >> 4) | (1u << 16);
      // V is MN-major: LBO = one box (the two 64-column halves of dv)
      const uint32_t v_lo = ((sbase + Ly::kKVOff + 3 * Ly::kKBox) >> 4) | ((Ly::kKBox >> 4) << 16);
      constexpr uint32_t kStageLo = Ly::kKVStage >> 4;
      uint32_t gq = 0, gk = 0, gs = 0, gt = 0;
      bool ok = true, issued = false;
      auto issue_pv = [&](uint32_t g, uint32_t st, bool first) -> bool {
        const uint32_t buf = g & 1;
        if (!wait_bar(B_PFULL(buf), (g >> 1) & 1, abort_flag, 4)) return false;
        tc_fence_after();
        if (first) {
          if (!wait_bar(B_OEMPTY, (gt & 1) ^ 1, abort_flag, 5)) return false;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts2(tmem + kDecTmemO, tmem + buf * BN + kk * 8, v_lo + st * kStageLo + kk * 128,
                  kDescHi, kIdPV, (!first || kk > 0) ? 1u : 0u);
        mma_commit(B_KVEMPTY(st));
        mma_commit(B_PVDONE);
        return true;
      };
      for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
        const Item it = make_item(args, w, BN);
        if (!it.valid) continue;
        if (!(ok = wait_bar(B_QREADY, gq & 1, abort_flag, 3))) break;
        tc_fence_after();
        for (int32_t j = 0; ok && j < it.n_blk; ++j) {
          const uint32_t st = (gk + j) % S;
          if (!(ok = wait_bar(B_KREADY(st), ((gk + j) / S) & 1, abort_flag, 6))) break;
          tc_fence_after();
          const uint32_t s_t = tmem + ((gs + j) & 1) * BN;
#pragma unroll
          for (int kstep = 0; kstep < kDqk / 16; ++kstep) {
            const uint32_t box = kstep >> 2, off = (kstep & 3) * 32;
            mma_ss2(s_t, q_lo + ((box * kQBoxBytes + off) >> 4), kDescHi,
                    kv_lo + st * kStageLo + ((box * Ly::kKBox + off) >> 4), kDescHi,
                    box == 0 ? kIdQKRot : kIdQK, kstep > 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit(B_SFULL((gs + j) & 1));
          if (j == it.n_blk - 1) mma_commit(B_QEMPTY);
          if (j > 0 && !(ok = issue_pv(gs + j - 1, (gk + j - 1) % S, j == 1))) break;
        }
        if (ok) ok = issue_pv(gs + it.n_blk - 1, (gk + it.n_blk - 1) % S, it.n_blk == 1);
        ++gq;
        gk += it.n_blk;
        gs += it.n_blk;
        ++gt;
      }
      if (issued) {
        mma_commit(B_DRAIN);
        drain_wait(B_DRAIN, 0);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ============================================================ online softmax
    const int32_t row = threadIdx.x - 128;  // packed row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool warp_active = (warp & 3) * 32 < R;  // the warp holds at least one real row
    const int32_t t = row / G, g = row % G;
    const float sc = args.scale_log2;
    const int32_t W = args.window;
    uint32_t gs = 0, gpv = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
      const Item it = make_item(args, w, BN);
      if (!it.valid) continue;
      // query t sits at position L - T + t and sees keys [max(0, pos - W + 1), pos]
      // of the cache, here limited to this chunk's keys [key_lo, key_hi)
      const int32_t pos = it.pos0 + t;
      const bool rvalid = row < R && pos >= 0;
      int32_t qlo = max(it.key_lo, W > 0 ? pos - W + 1 : 0);
      int32_t qhi = min(pos, it.key_hi - 1);
      if (!rvalid) { qlo = 1 << 30; qhi = 1 << 30; }
      float m = -INFINITY, l = 0.f;
      for (int32_t j = 0; ok && j < it.n_blk; ++j) {
        const uint32_t buf = gs & 1;
        if (!(ok = wait_bar_warp(B_SFULL(buf), (gs >> 1) & 1, abort_flag, 7))) break;
        tc_fence_after();
        bool alpha_any = false;
        float alpha_row = 1.f;
        if (warp_active) {
          const uint32_t s_t = tmem + lane_off + buf * BN;
          uint32_t r[BN];
          tmem_ld32p(s_t, r);
          tmem_ld32p(s_t + 32, r + 32);
          tmem_wait_ld();
          reg_fence<BN>(r);
          // visible columns of this block: k - lo <= span (unsigned)
          const int32_t kb = it.kstart + j * BN;
          const int32_t lo = qlo - kb;
          const uint32_t span = static_cast<uint32_t>(qhi - qlo);
          const bool whole = lo <= 0 && lo + static_cast<int32_t>(span) >= BN - 1;
          if (!__all_sync(0xffffffffu, whole)) {
#pragma unroll
            for (int32_t k = 0; k < BN; ++k)
              if (static_cast<uint32_t>(k - lo) > span) r[k] = 0xff800000u;  // -inf
          }
          float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
          for (int32_t k = 0; k < BN; k += 4) {
            mxa = fmax3(mxa, __uint_as_float(r[k]), __uint_as_float(r[k + 1]));
            mxb = fmax3(mxb, __uint_as_float(r[k + 2]), __uint_as_float(r[k + 3]));
          }
          const float mx = fmaxf(mxa, mxb) * sc;
          // lazy running max: move only when this block exceeds it by more
          // than 8 (P stays <= 2^8); the final normalisation uses the same m
          const float m_new = (mx > m + 8.f) ? mx : m;
          const float mneg = m_new == -INFINITY ? 0.f : -m_new;
          const float2 sc2 = make_float2(sc, sc), mneg2 = make_float2(mneg, mneg);
          float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int32_t k = 0; k < BN; k += 2) {
            const float2 y = ffma2(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                                   sc2, mneg2);
            const float2 p = make_float2(ex2(y.x), ex2(y.y));
            sum2 = fadd2(sum2, p);
            r[k >> 1] = pack_bf16x2(p.x, p.y);
          }
          tmem_st32p(s_t, r);  // P over the S columns already read
          const float alpha = (m_new == m) ? 1.f : ex2(m - m_new);
          l = l * alpha + (sum2.x + sum2.y);
          m = m_new;
          tmem_wait_st();
          alpha_any = __any_sync(0xffffffffu, alpha != 1.f);
          alpha_row = alpha;
        }
        // PV_DONE is consumed in order, once per block (a parity wait must not
        // fall two phases behind): S_FULL(j) implies PV(j-2) completed and PV(j)
        // needs this block's P, so phase j-1 is the only one in doubt here.
        if (j > 0) {
          if (!(ok = wait_bar_warp(B_PVDONE, (gpv + j - 1) & 1, abort_flag, 8))) break;
          tc_fence_after();
          if (alpha_any) {
            // the running max moved: rescale this row's O before PV(j) adds to it
            const uint32_t o_t = tmem + lane_off + kDecTmemO;
#pragma unroll 1
            for (int32_t c0 = 0; c0 < kDv; c0 += 32) {
              uint32_t o[32];
              tmem_ld32p(o_t + c0, o);
              tmem_wait_ld();
              reg_fence<32>(o);
#pragma unroll
              for (int32_t c = 0; c < 32; c += 2) {
                const float2 v = fmul2(make_float2(__uint_as_float(o[c]), __uint_as_float(o[c + 1])),
                                       make_float2(alpha_row, alpha_row));
                o[c] = __float_as_uint(v.x);
                o[c + 1] = __float_as_uint(v.y);
              }
              tmem_st32p(o_t + c0, o);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        mbar_arrive(B_PFULL(buf));
        ++gs;
      }
      if (!ok) break;
      // ---------------- the chunk's partial: unnormalised O, m and l (log2 domain)
      if (!(ok = wait_bar_warp(B_PVDONE, (gpv + it.n_blk - 1) & 1, abort_flag, 9))) break;
      gpv += it.n_blk;
      tc_fence_after();
      if (warp_active) {
        const uint32_t o_t = tmem + lane_off + kDecTmemO;
        const size_t prow = static_cast<size_t>(it.out_idx) * R + row;
        float4 *dst = reinterpret_cast<float4 *>(args.part_o + prow * kDv);
#pragma unroll 1
        for (int32_t c0 = 0; c0 < kDv; c0 += 32) {
          uint32_t o[32];
          tmem_ld32p(o_t + c0, o);
          tmem_wait_ld();
          reg_fence<32>(o);
          if (row < R) {
#pragma unroll
            for (int32_t q4 = 0; q4 < 8; ++q4)
              dst[c0 / 4 + q4] = make_float4(__uint_as_float(o[4 * q4]), __uint_as_float(o[4 * q4 + 1]),
                                             __uint_as_float(o[4 * q4 + 2]),
                                             __uint_as_float(o[4 * q4 + 3]));
          }
        }
        if (row < R) reinterpret_cast<float4 *>(args.part_ml)[prow] = make_float4(m, l, l, 0.f);
      }
      tc_fence_before();
      mbar_arrive(B_OEMPTY);
    }
  } else if (warp >= 8) {
    // ============================================================ RoPE
    const int32_t tid = threadIdx.x - 256;
    uint32_t gq = 0, gk = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
      const Item it = make_item(args, w, BN);
      if (!it.valid) continue;
      if (!(ok = wait_bar_warp(B_QFULL, gq & 1, abort_flag, 10))) break;
      if (args.rope_on)
        rope_q_tile(smem + Ly::kQOff, G, it.n_tok, it.pos0, args.rope_style, turns, tid);
      fence_proxy_async_smem();
      mbar_arrive(B_QREADY);
      ++gq;
      for (int32_t j = 0; j < it.n_blk; ++j) {
        const uint32_t st = gk % S;
        if (!(ok = wait_bar_warp(B_KVFULL(st), (gk / S) & 1, abort_flag, 11))) break;
        if (args.rope_on)
          rope_k_rows(smem + Ly::kKVOff + st * Ly::kKVStage, BN, it.kstart + j * BN, args.rope_style,
                      turns, tid);
        fence_proxy_async_smem();
        mbar_arrive(B_KREADY(st));
        ++gk;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kDecTmemCols);
  }
}

}  // namespace sa
