// attn_kernel.cuh -- the general sink-bias GQA prefill kernel for sm_103a.
//
// Prefill with a positive logit scale runs on specialised kernels
// (band_kernel.cuh: sliding window, 8 heads per KV head, W <= 128;
// causal_kernel.cuh: every other shape, global or windowed).  This kernel
// covers the rest: logit scales <= 0, whose running maximum it takes over the
// scaled logits.
//
// Computes, for one tile of 128 packed query rows at a time, the attention of
// the MiMo-V2-Flash Technical Report (§2.2 eqs. (1)-(3); shapes from §2.1
// Table 1):  a = q.k / sqrt(192) on RoPE-rotated q, k (first 64 dims),
// s = exp(a - m) / (exp(sink - m) + sum exp(a - m)), o = sum s v.
//
// Design (one persistent CTA per SM, 12 warps, warp-specialised):
//   warp 0       TMA producer: Q tile (3 boxes of 64 dims) and K/V blocks of
//                BN keys into shared-memory rings (128-byte swizzle).
//   warp 1       MMA issuer: S = Q K^T (tcgen05, bf16 -> fp32 in TMEM, 12 k-steps
//                of 16), then O += P V with P read from TMEM (aliasing S).
//   warp 2       TMEM allocator (512 columns: S0, S1, O).
//   warps 4-7    softmax + epilogue, one query row per thread (= TMEM lane):
//                online softmax whose running max starts AT THE SINK and whose
//                denominator starts at exp(sink - m) = 1, so the sink enters the
//                denominator exactly once (eq. (2)); lazy rescale of O.
//   warps 8-11   RoPE: rotate dims 0..63 of the Q tile and of every K block in
//                shared memory before the MMA reads them.
// GQA head packing: the 128 MMA rows are G query heads x (128 / G) tokens that
// share one KV head (row r = token * G + head), so every K/V block is loaded
// once for all G heads.
//
// Every wait is bounded: on expiry a CTA records SINKATTN_ETIMEOUT in the
// device status word, tells its other warps to stop, drains its own
// outstanding copies and MMAs, frees its TMEM and returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace sa {

struct AttnArgs {
  int32_t Hq, Hkv, G;
  int32_t tile_tokens;     // tokens per tile: 128 / G
  int32_t window;
  int32_t batch;
  int32_t n_items;         // virtual work items (some are empty and skipped)
  int32_t tiles_per_seq;   // ceil(max_seqlen / tile_tokens)
  int32_t lpt_order;       // 1: walk tiles longest-first (global causal prefill)
  int32_t rope_on, rope_style;
  uint32_t q_tx_bytes;     // bytes of one Q tile load (3 boxes)
  float scale_log2;        // logit scale * log2(e)
  const int32_t *cu_seqlens;
  const float *sink;
  __nv_bfloat16 *out;
  float *lse;
  int64_t n_rows;          // rows of out and lse: tokens x Hq (checked stores)
  unsigned long long rope_turns[32];  // round(theta_t / (2 pi) * 2^64), t = 0..31
};

// One work item: a tile of packed query rows and the key blocks it visits.
struct Item {
  int32_t valid;
  int32_t b, kvh;
  int32_t n_tok;    // valid tokens in the tile
  int32_t pos0;     // position of the tile's first token
  int32_t q_row;    // outer TMA coordinate of that token in the Q map
  int32_t kv_row0;  // outer TMA coordinate of key position 0 in the K/V maps
  int32_t kstart;   // key position of column 0 of block 0
  int32_t n_blk;
  int32_t key_lo, key_hi;  // keys this item may use: [key_lo, key_hi)
};

__device__ __forceinline__ Item make_item(const AttnArgs &a, int32_t w, int32_t BN) {
  Item it;
  it.valid = 0;
  int32_t i, r;
  if (a.lpt_order) {
    const int32_t per = a.batch * a.Hkv;
    i = a.tiles_per_seq - 1 - w / per;
    r = w % per;
  } else {
    i = w % a.tiles_per_seq;
    r = w / a.tiles_per_seq;
  }
  it.kvh = r % a.Hkv;
  it.b = r / a.Hkv;
  const int32_t s0 = __ldg(a.cu_seqlens + it.b);
  const int32_t L = __ldg(a.cu_seqlens + it.b + 1) - s0;
  it.pos0 = i * a.tile_tokens;
  if (it.pos0 >= L) return it;
  it.n_tok = min(a.tile_tokens, L - it.pos0);
  it.q_row = s0 + it.pos0;
  it.kv_row0 = s0;
  const int32_t hi = it.pos0 + it.n_tok;
  it.kstart = a.window > 0 ? max(0, it.pos0 - a.window + 1) : 0;
  it.n_blk = (hi - it.kstart + BN - 1) / BN;
  it.key_lo = 0;
  it.key_hi = hi;
  it.valid = 1;
  return it;
}

template <int BN, int NQ, int NKV>
struct Layout {
  static constexpr uint32_t kKBox = BN * kRowBytes;
  static constexpr uint32_t kKVStage = 5 * kKBox;  // K: 3 boxes, V: 2 boxes
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = NQ * kQStageBytes;
  static constexpr uint32_t kBarOff = kKVOff + NKV * kKVStage;
  // barriers: q_full, q_ready, q_empty [NQ]; kv_full, k_ready, kv_empty [NKV];
  // s_full[2], p_full[2], pv_done, o_empty, drain
  static constexpr uint32_t kNumBars = 3 * NQ + 3 * NKV + 7;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kTurnsOff = (kMiscOff + 16 + 7) & ~7u;
  static constexpr uint32_t kBytes = kTurnsOff + 32 * 8;
  static constexpr uint32_t kDynSmem = kBytes + 1024;  // slack for 1024-byte alignment
};

template <int BN, int NQ, int NKV>
__global__ void __launch_bounds__(kThreads, 1)
    sinkattn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ AttnArgs args) {
  using Ly = Layout<BN, NQ, NKV>;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 192, "key block size");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);

  const int32_t warp = threadIdx.x >> 5;
  const int32_t lane = threadIdx.x & 31;

  auto bar = [&](uint32_t i) { return sbase + Ly::kBarOff + i * 8; };
  auto B_QFULL = [&](uint32_t s) { return bar(s); };
  auto B_QREADY = [&](uint32_t s) { return bar(NQ + s); };
  auto B_QEMPTY = [&](uint32_t s) { return bar(2 * NQ + s); };
  auto B_KVFULL = [&](uint32_t s) { return bar(3 * NQ + s); };
  auto B_KREADY = [&](uint32_t s) { return bar(3 * NQ + NKV + s); };
  auto B_KVEMPTY = [&](uint32_t s) { return bar(3 * NQ + 2 * NKV + s); };
  auto B_SFULL = [&](uint32_t b) { return bar(3 * NQ + 3 * NKV + b); };
  auto B_PFULL = [&](uint32_t b) { return bar(3 * NQ + 3 * NKV + 2 + b); };
  const uint32_t B_PVDONE = bar(3 * NQ + 3 * NKV + 4);
  const uint32_t B_OEMPTY = bar(3 * NQ + 3 * NKV + 5);
  const uint32_t B_DRAIN = bar(3 * NQ + 3 * NKV + 6);

  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  unsigned long long *turns = reinterpret_cast<unsigned long long *>(smem + Ly::kTurnsOff);

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < NQ; ++s) {
      mbar_init(B_QFULL(s), 1);
      mbar_init(B_QREADY(s), 128);
      mbar_init(B_QEMPTY(s), 1);
    }
    for (uint32_t s = 0; s < NKV; ++s) {
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
    tmem_alloc(sbase + Ly::kMiscOff, kTmemCols);
    tmem_relinquish();
  }
  // Zero the Q stages once: decode tiles fill fewer than 128 rows and the
  // MMA reads all 128 (padding rows must hold finite values).
  for (uint32_t i = threadIdx.x; i < NQ * kQStageBytes / 16; i += kThreads)
    reinterpret_cast<uint4 *>(smem + Ly::kQOff)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int32_t G = args.G;
  const int32_t W = args.window;

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
        const uint32_t qs = gq % NQ;
        if (!(ok = wait_bar(B_QEMPTY(qs), ((gq / NQ) & 1) ^ 1, abort_flag, 1))) break;
        mbar_arrive_expect_tx(B_QFULL(qs), args.q_tx_bytes);
        const uint32_t qdst = sbase + Ly::kQOff + qs * kQStageBytes;
#pragma unroll
        for (int c = 0; c < 3; ++c)
          tma_load_3d(qdst + c * kQBoxBytes, &tm_q, c * 64, it.kvh * G, it.q_row, B_QFULL(qs));
        ++gq;
        for (int32_t j = 0; j < it.n_blk; ++j) {
          const uint32_t ks = gk % NKV;
          if (!(ok = wait_bar(B_KVEMPTY(ks), ((gk / NKV) & 1) ^ 1, abort_flag, 2))) break;
          mbar_arrive_expect_tx(B_KVFULL(ks), Ly::kKVStage);
          const uint32_t kdst = sbase + Ly::kKVOff + ks * Ly::kKVStage;
          const int32_t krow = it.kv_row0 + it.kstart + j * BN;
#pragma unroll
          for (int c = 0; c < 3; ++c)
            tma_load_3d(kdst + c * Ly::kKBox, &tm_k, c * 64, it.kvh, krow, B_KVFULL(ks));
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_3d(kdst + (3 + c) * Ly::kKBox, &tm_v, c * 64, it.kvh, krow, B_KVFULL(ks));
          ++gk;
        }
      }
      // Drain: the last copy into each stage must have landed before the CTA exits.
      for (uint32_t s = 0; s < NQ; ++s)
        if (gq > s) drain_wait(B_QFULL(s), ((gq - 1 - s) / NQ) & 1);
      for (uint32_t s = 0; s < NKV; ++s)
        if (gk > s) drain_wait(B_KVFULL(s), ((gk - 1 - s) / NKV) & 1);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_f32acc(128, BN, 1, 0, 0);
      constexpr uint32_t kIdescQKRot = idesc_f32acc(128, BN, 0, 0, 0);  // fp16 rotated dims
      constexpr uint32_t kIdescPV = idesc_f32acc(128, kDv, 1, 0, 1);
      const uint32_t idesc_box0 = args.rope_on ? kIdescQKRot : kIdescQK;
      uint32_t gq = 0, gk = 0, gs = 0, gt = 0;
      bool ok = true, issued = false;
      for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
        const Item it = make_item(args, w, BN);
        if (!it.valid) continue;
        const uint32_t qs = gq % NQ;
        if (!(ok = wait_bar(B_QREADY(qs), (gq / NQ) & 1, abort_flag, 3))) break;
        tc_fence_after();
        const uint32_t qaddr = sbase + Ly::kQOff + qs * kQStageBytes;

        auto issue_pv = [&](int32_t jj) -> bool {
          const uint32_t g = gs + jj;
          const uint32_t buf = g & 1;
          if (!wait_bar(B_PFULL(buf), (g >> 1) & 1, abort_flag, 4)) return false;
          tc_fence_after();
          if (jj == 0) {
            if (!wait_bar(B_OEMPTY, (gt & 1) ^ 1, abort_flag, 5)) return false;
            tc_fence_after();
          }
          const uint32_t ks = (gk + jj) % NKV;
          const uint32_t vaddr = sbase + Ly::kKVOff + ks * Ly::kKVStage + 3 * Ly::kKBox;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            // B = V rows (keys) kk*16 .. kk*16+15, MN-major: the two 64-column
            // halves of dv are LBO = one box apart, 8-key groups SBO = 1024 B apart.
            const uint64_t bdesc = smem_desc_sw128(vaddr + kk * 16 * kRowBytes, Ly::kKBox, 1024);
            mma_ts(tmem + kTmemO, tmem + tmem_s_col(buf) + kk * 8, bdesc, kIdescPV,
                   (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(B_KVEMPTY(ks));
          mma_commit(B_PVDONE);
          return true;
        };

        for (int32_t j = 0; ok && j < it.n_blk; ++j) {
          if (NKV == 1 && j > 0) {
            if (!(ok = issue_pv(j - 1))) break;
          }
          const uint32_t gkj = gk + j;
          const uint32_t ks = gkj % NKV;
          if (!(ok = wait_bar(B_KREADY(ks), (gkj / NKV) & 1, abort_flag, 6))) break;
          tc_fence_after();
          const uint32_t buf = (gs + j) & 1;
          const uint32_t kaddr = sbase + Ly::kKVOff + ks * Ly::kKVStage;
#pragma unroll
          for (int kstep = 0; kstep < kDqk / 16; ++kstep) {
            const uint32_t box = kstep >> 2, off = (kstep & 3) * 32;
            const uint64_t adesc = smem_desc_sw128(qaddr + box * kQBoxBytes + off, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(kaddr + box * Ly::kKBox + off, 16, 1024);
            mma_ss(tmem + tmem_s_col(buf), adesc, bdesc, box == 0 ? idesc_box0 : kIdescQK,
                   kstep > 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit(B_SFULL(buf));
          if (j == it.n_blk - 1) mma_commit(B_QEMPTY(qs));
          if (NKV > 1 && j > 0) {
            if (!(ok = issue_pv(j - 1))) break;
          }
        }
        if (ok) ok = issue_pv(it.n_blk - 1);
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
    // ============================================================ softmax + epilogue
    const int32_t row = threadIdx.x - 128;  // query row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t gs = 0, gp = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
      const Item it = make_item(args, w, BN);
      if (!it.valid) continue;
      const int32_t t = row / G, g = row % G;
      const int32_t head = it.kvh * G + g;
      const bool rvalid = t < it.n_tok;
      const int32_t pos = it.pos0 + t;
      int32_t lo = max(it.key_lo, W > 0 ? pos - W + 1 : 0);
      int32_t hi = min(pos, it.key_hi - 1);
      if (!rvalid) { lo = 1; hi = 0; }
      // Running max starts at the sink and the denominator at exp(sink - m) = 1
      // (eq. (2)); a -inf sink starts from the empty sum.  Two denominators are
      // kept: `l` sums the fp32 weights (for lse), `lr` sums the bf16-rounded
      // weights that the PV MMA actually multiplies, so O / lr cancels the
      // rounding of P.
      float m = -INFINITY, l = 0.f, lr = 0.f;
      {
        const float sk = __ldg(args.sink + head);
        if (sk != -INFINITY) { m = sk * kLog2e; l = 1.f; lr = 1.f; }
      }
      for (int32_t j = 0; ok && j < it.n_blk; ++j) {
        const uint32_t buf = gs & 1;
        if (!(ok = wait_bar_warp(B_SFULL(buf), (gs >> 1) & 1, abort_flag, 7))) break;
        tc_fence_after();
        const uint32_t s_t = tmem + lane_off + tmem_s_col(buf);
        const int32_t kb = it.kstart + j * BN;
        // pass 1: the block's row max of the scaled, masked logits (log2 domain)
        float mx = -INFINITY;
#pragma unroll
        for (int32_t c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          if (BN - c0 >= 32) tmem_ld32(s_t + c0, r); else tmem_ld16(s_t + c0, r);
          tmem_wait_ld();
          reg_fence<32>(r);
#pragma unroll
          for (int32_t c = 0; c < 32; ++c) {
            if (c0 + c < BN) {
              const int32_t kp = kb + c0 + c;
              const float x = __uint_as_float(r[c]) * args.scale_log2;
              if (kp >= lo && kp <= hi) mx = fmaxf(mx, x);
            }
          }
        }
        // Lazy max: move m only when the block max exceeds it by more than 8
        // (P stays <= 2^8); the final normalisation uses the same m.
        const float m_new = (mx > m + 8.f) ? mx : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (m_new == m) ? 1.f : ex2(m - m_new);
        // pass 2: P = 2^(x - m) as bf16 into TMEM over the consumed S columns
        float sum = 0.f, sum_r = 0.f;
#pragma unroll
        for (int32_t c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          const bool full = BN - c0 >= 32;
          if (full) tmem_ld32(s_t + c0, r); else tmem_ld16(s_t + c0, r);
          tmem_wait_ld();
          reg_fence<32>(r);
          uint32_t pk[16];
#pragma unroll
          for (int32_t c = 0; c < 32; c += 2) {
            if (c0 + c < BN) {
              const int32_t kp = kb + c0 + c;
              const float x0 = __uint_as_float(r[c]) * args.scale_log2;
              const float x1 = __uint_as_float(r[c + 1]) * args.scale_log2;
              const float p0 = (kp >= lo && kp <= hi) ? ex2(x0 - m_use) : 0.f;
              const float p1 = (kp + 1 >= lo && kp + 1 <= hi) ? ex2(x1 - m_use) : 0.f;
              const uint32_t pw = pack_bf16x2(p0, p1);
              sum += p0 + p1;
              sum_r += bf16lo(pw) + bf16hi(pw);
              pk[c >> 1] = pw;
            }
          }
          if (full) tmem_st16(s_t + c0 / 2, pk); else tmem_st8(s_t + c0 / 2, pk);
        }
        tmem_wait_st();
        l = l * alpha + sum;
        lr = lr * alpha + sum_r;
        m = m_new;
        if (j > 0) {
          // the previous block's PV has to land before O may be rescaled
          if (!(ok = wait_bar_warp(B_PVDONE, gp & 1, abort_flag, 8))) break;
          ++gp;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            const uint32_t o_t = tmem + lane_off + kTmemO;
#pragma unroll
            for (int32_t c0 = 0; c0 < kDv; c0 += 32) {
              uint32_t r[32];
              tmem_ld32(o_t + c0, r);
              tmem_wait_ld();
              reg_fence<32>(r);
#pragma unroll
              for (int32_t c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
              tmem_st32(o_t + c0, r);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        mbar_arrive(B_PFULL(buf));
        ++gs;
      }
      if (!ok) break;
      // ---------------- epilogue: O / l and lse
      if (!(ok = wait_bar_warp(B_PVDONE, gp & 1, abort_flag, 9))) break;
      ++gp;
      tc_fence_after();
      const uint32_t o_t = tmem + lane_off + kTmemO;
      const float inv_l = lr > 0.f ? 1.f / lr : 0.f;
      const size_t orow = static_cast<size_t>(it.q_row + t) * args.Hq + head;
      uint4 *dst = reinterpret_cast<uint4 *>(args.out + orow * kDv);
      const bool st_ok = rvalid && SA_OUT(orow, args.n_rows, 0x10);
#pragma unroll
      for (int32_t c0 = 0; c0 < kDv; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(o_t + c0, r);
        tmem_wait_ld();
        reg_fence<32>(r);
        if (st_ok) {
#pragma unroll
          for (int32_t q4 = 0; q4 < 4; ++q4) {
            uint32_t w4[4];
#pragma unroll
            for (int32_t e = 0; e < 4; ++e)
              w4[e] = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2 * e]) * inv_l,
                                  __uint_as_float(r[q4 * 8 + 2 * e + 1]) * inv_l);
            dst[c0 / 8 + q4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      if (st_ok) args.lse[orow] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
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
      const uint32_t qs = gq % NQ;
      if (!(ok = wait_bar_warp(B_QFULL(qs), (gq / NQ) & 1, abort_flag, 10))) break;
      if (args.rope_on)
        rope_q_tile(smem + Ly::kQOff + qs * kQStageBytes, G, it.n_tok, it.pos0, args.rope_style,
                    turns, tid);
      fence_proxy_async_smem();
      mbar_arrive(B_QREADY(qs));
      ++gq;
      for (int32_t j = 0; j < it.n_blk; ++j) {
        const uint32_t ks = gk % NKV;
        if (!(ok = wait_bar_warp(B_KVFULL(ks), (gk / NKV) & 1, abort_flag, 11))) break;
        if (args.rope_on)
          rope_k_rows(smem + Ly::kKVOff + ks * Ly::kKVStage, BN, it.kstart + j * BN,
                      args.rope_style, turns, tid);
        fence_proxy_async_smem();
        mbar_arrive(B_KREADY(ks));
        ++gk;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace sa
