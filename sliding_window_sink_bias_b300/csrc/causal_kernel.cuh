// causal_kernel.cuh -- global causal (GA) prefill, two query tiles per CTA.
//
// Computes the attention layer of the MiMo-V2-Flash Technical Report (§2.2
// eqs. (1)-(3), shapes of §2.1 Table 1) for the global layers: every query
// attends to all keys at or before its position, with the per-head sink in the
// softmax denominator.  The same kernel runs the sliding windows the band
// kernel does not take (window > 128, or other than 8 query heads per KV
// head): an item then visits only the 128-key blocks its window reaches, and
// the low edge of the window is masked like the diagonal.
//
// A query tile is T = 128 / G consecutive tokens x the G query heads of one KV
// head (128 MMA rows, row r = token * G + head).  Each work item is a pair of
// adjacent tiles A and B of one (sequence, KV head); the pair shares every
// 128-key K/V block it loads (keys 0 .. end of tile B), so K/V traffic into
// shared memory and the K rotation are paid once per two tiles.  Items are
// visited longest first, so the persistent CTAs finish together.
//
// TMEM (512 columns): S_A, S_B (fp32 logits; P as bf16 pairs over their first
// 64 columns), O_A, O_B (fp32 accumulators).  The MMA issuer keeps the tensor
// pipe busy while each tile's softmax runs: per block j it issues
//   PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1),
// so the softmax of A overlaps PV_B and QK_B and vice versa.
//
// Warp roles (512 threads, one CTA per SM):
//   warp 0       TMA producer: the two Q tiles of an item, K blocks (2 stages).
//   warp 1       MMA issuer.
//   warp 2       TMEM allocator.
//   warp 3       TMA producer of V blocks (1 stage).
//   warps 4-7    softmax of tile A, warps 8-11 softmax of tile B: one row per
//                thread; per block the masked max (3-input max, chunks of 64
//                columns), a lazy running max (moves only when a block exceeds
//                it by more than 2^8; O is then rescaled), P = 2^(s * scale *
//                log2e - m), l; at the end o = O / l with the sink counted once,
//                and the log-sum-exp.
//   warps 12-15  RoPE on dims 0..63 of the Q tiles and of every K block.
#pragma once
#include "common.cuh"

namespace sa {

constexpr int32_t kCauBN = 128;       // keys per block
constexpr int32_t kCauThreads = 512;

struct CausalArgs {
  int32_t Hq, Hkv, G;
  int32_t window;       // 0: global causal; W > 0: keys (pos - W, pos]
  int32_t T;            // tokens per tile = 128 / G
  int32_t batch;
  int32_t max_seqlen;
  int32_t npairs;       // ceil(max_seqlen / (2 T))
  int32_t n_items;      // batch * Hkv * npairs (some are empty)
  int32_t rope_on, rope_style;
  uint32_t q_tx_bytes;  // one Q tile (3 boxes)
  float scale_log2;     // > 0
  int32_t out_v8;       // out is 32-byte aligned
  const int32_t *cu_seqlens;
  const float *sink;
  __nv_bfloat16 *out;
  float *lse;
  int64_t n_rows;       // rows of out and lse: tokens x Hq (checked stores)
  unsigned long long rope_turns[32];
};

struct CauLayout {
  static constexpr uint32_t kKBox = kCauBN * kRowBytes;    // 128 keys x 64 dims: 16 KB
  static constexpr uint32_t kQOff = 0;                     // tiles A, B: 2 x 48 KB
  static constexpr uint32_t kKOff = 2 * kQStageBytes;      // 2 stages x 3 boxes
  static constexpr uint32_t kKStage = 3 * kKBox;
  static constexpr uint32_t kVOff = kKOff + 2 * kKStage;   // 1 stage x 2 boxes
  static constexpr uint32_t kBarOff = kVOff + 2 * kKBox;
  // q_full[2] q_ready[2] q_empty | k_full[2] k_ready[2] k_empty[2] | v_full v_empty |
  // s_full[2] p_full[2] pv_done[2] o_empty[2] | drain
  static constexpr uint32_t kNumBars = 5 + 6 + 2 + 8 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;  // tmem slot, abort flag
  static constexpr uint32_t kTurnsOff = (kMiscOff + 16 + 7) & ~7u;
  static constexpr uint32_t kBytes = kTurnsOff + 32 * 8;
  static constexpr uint32_t kDynSmem = kBytes + 1024;
};
static_assert(CauLayout::kDynSmem <= 232448, "causal kernel shared memory");

// One work item: tiles A and B = tokens [t0, t0 + 2T) of sequence b, KV head kvh.
struct CauItem {
  int32_t valid;
  int32_t b, kvh;
  int32_t s0, L;   // first packed row and length of the sequence
  int32_t t0;      // position of tile A's first token
  int32_t kb0;     // first key block: the one holding key max(0, t0 - W + 1) (0 if global)
  int32_t nblk;    // key blocks kb0 .. kb0 + nblk - 1: keys up to min(L, t0 + 2T) - 1
};

// Items longest first: pair index descending, then (sequence, KV head).
__device__ __forceinline__ CauItem cau_item(const CausalArgs &a, int32_t w) {
  CauItem it;
  const int32_t per = a.batch * a.Hkv;
  const int32_t n = a.npairs - 1 - w / per;
  const int32_t r = w % per;
  it.kvh = r % a.Hkv;
  it.b = r / a.Hkv;
  it.s0 = __ldg(a.cu_seqlens + it.b);
  it.L = __ldg(a.cu_seqlens + it.b + 1) - it.s0;
  it.t0 = n * 2 * a.T;
  it.valid = it.t0 < it.L;
  const int32_t kend = min(it.L, it.t0 + 2 * a.T);
  it.kb0 = a.window > 0 ? max(0, it.t0 - a.window + 1) / kCauBN : 0;
  it.nblk = (kend + kCauBN - 1) / kCauBN - it.kb0;
  return it;
}

// Softmax + epilogue of one tile (X = 0: A, 1: B) of every item; one row per thread.
__device__ __forceinline__ void cau_softmax(const CausalArgs &args, int32_t X, uint32_t tmem,
                                            uint32_t sbase, volatile uint32_t *abort_flag) {
  using Ly = CauLayout;
  const uint32_t bars = sbase + Ly::kBarOff;
  const uint32_t B_SFULL = bars + (13 + X) * 8;
  const uint32_t B_PFULL = bars + (15 + X) * 8;
  const uint32_t B_PVDONE = bars + (17 + X) * 8;
  const uint32_t B_OEMPTY = bars + (19 + X) * 8;
  const int32_t warp = threadIdx.x >> 5;
  const int32_t row = (warp & 3) * 32 + (threadIdx.x & 31);  // query row == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t s_t = tmem + lane_off + X * 128;
  const uint32_t o_t = tmem + lane_off + 256 + X * 128;
  const int32_t G = args.G;
  const int32_t t = row / G, g = row % G;
  const float sc = args.scale_log2;
  constexpr uint32_t kNegInf = 0xff800000u;
  uint32_t gb = 0;  // blocks seen (S_FULL / P_FULL / PV_DONE phases)
  uint32_t gi = 0;  // items seen (O_EMPTY phases)
  bool ok = true;
  for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
    const CauItem it = cau_item(args, w);
    if (!it.valid) continue;
    const int32_t pos = it.t0 + X * args.T + t;  // this row's position
    const bool rvalid = pos < it.L;
    const int32_t head = it.kvh * G + g;
    float m = -INFINITY, l = 0.f;
    for (int32_t j = 0; ok && j < it.nblk; ++j) {
      if (!(ok = wait_bar_warp(B_SFULL, gb & 1, abort_flag, 7))) break;
      tc_fence_after();
      // visible columns of block j (keys from 128 (kb0 + j)): lo <= k <= hi,
      // lo from the window (none for a padding row)
      const int32_t kbase = (it.kb0 + j) * kCauBN;
      const int32_t hi = rvalid ? pos - kbase : -1;
      const int32_t lo = args.window > 0 ? pos - args.window + 1 - kbase : INT32_MIN;
      const bool whole = __all_sync(0xffffffffu, hi >= kCauBN - 1 && lo <= 0);
      float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll 1
      for (int32_t ch = 0; ch < 2; ++ch) {
        uint32_t r[64];
        tmem_ld32p(s_t + ch * 64, r);
        tmem_ld32p(s_t + ch * 64 + 32, r + 32);
        tmem_wait_ld();
        reg_fence<64>(r);
        if (!whole) {
          // masked columns become -inf in TMEM too, so the exp pass needs no mask
#pragma unroll
          for (int32_t k = 0; k < 64; ++k)
            if (ch * 64 + k > hi || ch * 64 + k < lo) r[k] = kNegInf;
          tmem_st32p(s_t + ch * 64, r);
          tmem_st32p(s_t + ch * 64 + 32, r + 32);
        }
#pragma unroll
        for (int32_t k = 0; k < 64; k += 4) {
          mxa = fmax3(mxa, __uint_as_float(r[k]), __uint_as_float(r[k + 1]));
          mxb = fmax3(mxb, __uint_as_float(r[k + 2]), __uint_as_float(r[k + 3]));
        }
      }
      if (!whole) tmem_wait_st();
      const float mx = fmaxf(mxa, mxb) * sc;
      // lazy running max: move only when this block exceeds it by more than 8
      // (P stays <= 2^8); the final normalisation uses the same m
      const float m_new = (mx > m + 8.f) ? mx : m;
      const float mneg = m_new == -INFINITY ? 0.f : -m_new;
      const float2 sc2 = make_float2(sc, sc), mneg2 = make_float2(mneg, mneg);
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int32_t ch = 0; ch < 2; ++ch) {
        uint32_t r[64];
        tmem_ld32p(s_t + ch * 64, r);
        tmem_ld32p(s_t + ch * 64 + 32, r + 32);
        tmem_wait_ld();
        reg_fence<64>(r);
#pragma unroll
        for (int32_t k = 0; k < 64; k += 2) {
          const float2 y = ffma2(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), sc2,
                                 mneg2);
          const float2 p = make_float2(ex2(y.x), ex2(y.y));
          sum2 = fadd2(sum2, p);
          r[k >> 1] = pack_bf16x2(p.x, p.y);
        }
        // P of columns 64 ch .. 64 ch + 63 -> TMEM columns 32 ch .. 32 ch + 31
        // (already read)
        tmem_st32p(s_t + ch * 32, r);
      }
      const float alpha = (m_new == m) ? 1.f : ex2(m - m_new);
      l = l * alpha + (sum2.x + sum2.y);
      m = m_new;
      tmem_wait_st();
      // S_FULL(j) was committed after PV(j-1), so O holds every earlier block
      // and the rescale needs no wait; PV_DONE is still consumed in order.
      if (j > 0) {
        if (!(ok = wait_bar_warp(B_PVDONE, (gb - 1) & 1, abort_flag, 8))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int32_t cb = 0; cb < kDv; cb += 32) {
            uint32_t o[32];
            tmem_ld32p(o_t + cb, o);
            tmem_wait_ld();
            reg_fence<32>(o);
#pragma unroll
            for (int32_t k = 0; k < 32; k += 2) {
              const float2 v = fmul2(make_float2(__uint_as_float(o[k]), __uint_as_float(o[k + 1])),
                                     make_float2(alpha, alpha));
              o[k] = __float_as_uint(v.x);
              o[k + 1] = __float_as_uint(v.y);
            }
            tmem_st32p(o_t + cb, o);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(B_PFULL);
      ++gb;
    }
    if (!ok) break;
    // ---------------- epilogue: o = O / L, L = l 2^(m - M) + 2^(sink - M), M = max(m, sink)
    if (!(ok = wait_bar_warp(B_PVDONE, (gb - 1) & 1, abort_flag, 9))) break;
    tc_fence_after();
    const float sk2 = __ldg(args.sink + head) * kLog2e;
    const float M = fmaxf(m, sk2);
    float scale_o = 0.f, lse_v = -INFINITY;
    if (M != -INFINITY) {
      const float a1 = m == -INFINITY ? 0.f : ex2(m - M);
      const float a2 = sk2 == -INFINITY ? 0.f : ex2(sk2 - M);
      const float Lw = l * a1 + a2;
      scale_o = a1 / Lw;
      lse_v = (M + __log2f(Lw)) * kLn2;
    }
    const size_t orow = static_cast<size_t>(it.s0 + pos) * args.Hq + head;
    const int32_t q = threadIdx.x & 3;
#pragma unroll 1
    for (int32_t hf = 0; hf < 2; ++hf) {
      uint32_t w[32];  // 64 output dims as bf16 pairs: four 32-byte sectors
      {
        uint32_t o[64];
        tmem_ld32p(o_t + hf * 64, o);
        tmem_ld32p(o_t + hf * 64 + 32, o + 32);
        tmem_wait_ld();
        reg_fence<64>(o);
        if (hf == 1) {
          // O is in registers: the next item's PV may overwrite it
          tc_fence_before();
          mbar_arrive(B_OEMPTY);
        }
#pragma unroll
        for (int32_t e = 0; e < 32; ++e) {
          const float2 v = fmul2(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])),
                                 make_float2(scale_o, scale_o));
          w[e] = pack_bf16x2(v.x, v.y);
        }
      }
      // Transpose the 4 x 4 sectors within each lane quad so each store writes
      // the whole 128-byte line of one of the quad's rows.
#pragma unroll
      for (int32_t jj = 0; jj < 2; ++jj) {
#pragma unroll
        for (int32_t e = 0; e < 8; ++e) {
          const uint32_t send = (q & 2) ? w[8 * jj + e] : w[8 * (jj + 2) + e];
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
          if (q & 2) w[8 * jj + e] = recv; else w[8 * (jj + 2) + e] = recv;
        }
      }
#pragma unroll
      for (int32_t jj = 0; jj < 4; jj += 2) {
#pragma unroll
        for (int32_t e = 0; e < 8; ++e) {
          const uint32_t send = (q & 1) ? w[8 * jj + e] : w[8 * (jj + 1) + e];
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
          if (q & 1) w[8 * jj + e] = recv; else w[8 * (jj + 1) + e] = recv;
        }
      }
      // The quad's rows are four heads of one token when G >= 4 (consecutive
      // rows of out), else the heads of two (G = 2) or four (G = 1) tokens.
#pragma unroll
      for (int32_t pq = 0; pq < 4; ++pq) {
        uint32_t (&sec)[8] = *reinterpret_cast<uint32_t(*)[8]>(w + 8 * pq);
        const int32_t rq = (row & ~3) + pq;
        const int32_t pos_q = it.t0 + X * args.T + rq / G;
        if (pos_q >= it.L) continue;
        const size_t orq = static_cast<size_t>(it.s0 + pos_q) * args.Hq + it.kvh * G + rq % G;
        if (!SA_OUT(orq, args.n_rows, 0x13)) continue;
        __nv_bfloat16 *dst = args.out + orq * kDv + hf * 64 + q * 16;
        if (args.out_v8) {
          st_global_v8(dst, sec);
        } else {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst);
          d4[0] = make_uint4(sec[0], sec[1], sec[2], sec[3]);
          d4[1] = make_uint4(sec[4], sec[5], sec[6], sec[7]);
        }
      }
    }
    if (rvalid && SA_OUT(orow, args.n_rows, 0x14)) args.lse[orow] = lse_v;
    ++gi;
  }
}

__global__ void __launch_bounds__(kCauThreads, 1)
    sinkattn_causal_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CausalArgs args) {
  using Ly = CauLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int32_t warp = threadIdx.x >> 5;
  const int32_t lane = threadIdx.x & 31;

  auto bar = [&](uint32_t i) { return sbase + Ly::kBarOff + i * 8; };
  auto B_QFULL = [&](uint32_t x) { return bar(x); };
  auto B_QREADY = [&](uint32_t x) { return bar(2 + x); };
  const uint32_t B_QEMPTY = bar(4);
  auto B_KFULL = [&](uint32_t s) { return bar(5 + s); };
  auto B_KREADY = [&](uint32_t s) { return bar(7 + s); };
  auto B_KEMPTY = [&](uint32_t s) { return bar(9 + s); };
  const uint32_t B_VFULL = bar(11), B_VEMPTY = bar(12);
  auto B_SFULL = [&](uint32_t x) { return bar(13 + x); };
  auto B_PFULL = [&](uint32_t x) { return bar(15 + x); };
  auto B_PVDONE = [&](uint32_t x) { return bar(17 + x); };
  auto B_OEMPTY = [&](uint32_t x) { return bar(19 + x); };
  const uint32_t B_DRAIN = bar(21);

  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  unsigned long long *turns = reinterpret_cast<unsigned long long *>(smem + Ly::kTurnsOff);

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (uint32_t x = 0; x < 2; ++x) {
      mbar_init(B_QFULL(x), 1);
      mbar_init(B_QREADY(x), 128);
      mbar_init(B_KFULL(x), 1);
      mbar_init(B_KREADY(x), 128);
      mbar_init(B_KEMPTY(x), 1);
      mbar_init(B_SFULL(x), 1);
      mbar_init(B_PFULL(x), 128);
      mbar_init(B_PVDONE(x), 1);
      mbar_init(B_OEMPTY(x), 128);
    }
    mbar_init(B_QEMPTY, 1);
    mbar_init(B_VFULL, 1);
    mbar_init(B_VEMPTY, 1);
    mbar_init(B_DRAIN, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) turns[threadIdx.x] = args.rope_turns[threadIdx.x];
  if (warp == 2) {
    tmem_alloc(sbase + Ly::kMiscOff, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int32_t G = args.G;

  if (warp == 0) {
    // ============================================================ TMA producer: Q, K
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      uint32_t gi = 0, gk = 0;
      bool ok = true;
      for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
        const CauItem it = cau_item(args, w);
        if (!it.valid) continue;
        if (!(ok = wait_bar(B_QEMPTY, (gi & 1) ^ 1, abort_flag, 1))) break;
        for (int32_t x = 0; x < 2; ++x) {
          mbar_arrive_expect_tx(B_QFULL(x), args.q_tx_bytes);
          const int32_t qrow = it.s0 + it.t0 + x * args.T;
#pragma unroll
          for (int cc = 0; cc < 3; ++cc)
            tma_load_3d(sbase + Ly::kQOff + x * kQStageBytes + cc * kQBoxBytes, &tm_q, cc * 64,
                        it.kvh * G, qrow, B_QFULL(x));
        }
        ++gi;
        for (int32_t j = 0; j < it.nblk; ++j) {
          const uint32_t st = gk & 1;
          if (!(ok = wait_bar(B_KEMPTY(st), ((gk >> 1) & 1) ^ 1, abort_flag, 2))) break;
          mbar_arrive_expect_tx(B_KFULL(st), Ly::kKStage);
#pragma unroll
          for (int cc = 0; cc < 3; ++cc)
            tma_load_3d(sbase + Ly::kKOff + st * Ly::kKStage + cc * Ly::kKBox, &tm_k, cc * 64,
                        it.kvh, it.s0 + (it.kb0 + j) * kCauBN, B_KFULL(st));
          ++gk;
        }
      }
      for (uint32_t x = 0; x < 2; ++x)
        if (gi > 0) drain_wait(B_QFULL(x), (gi - 1) & 1);
      for (uint32_t s = 0; s < 2; ++s)
        if (gk > s) drain_wait(B_KFULL(s), ((gk - 1 - s) >> 1) & 1);
    }
  } else if (warp == 3) {
    // ============================================================ TMA producer: V
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      uint32_t gv = 0;
      bool ok = true;
      for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
        const CauItem it = cau_item(args, w);
        if (!it.valid) continue;
        for (int32_t j = 0; j < it.nblk; ++j) {
          if (!(ok = wait_bar(B_VEMPTY, (gv & 1) ^ 1, abort_flag, 12))) break;
          mbar_arrive_expect_tx(B_VFULL, 2 * Ly::kKBox);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            tma_load_3d(sbase + Ly::kVOff + cc * Ly::kKBox, &tm_v, cc * 64, it.kvh,
                        it.s0 + (it.kb0 + j) * kCauBN, B_VFULL);
          ++gv;
        }
      }
      if (gv > 0) drain_wait(B_VFULL, (gv - 1) & 1);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t rot = args.rope_on ? 0u : 1u;  // rotated dims are fp16
      const uint32_t kIdQK = idesc_f32acc(128, kCauBN, 1, 0, 0);
      const uint32_t kIdQKRot = idesc_f32acc(128, kCauBN, rot, 0, 0);
      constexpr uint32_t kIdPV = idesc_f32acc(128, kDv, 1, 0, 1);
      constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
      const uint32_t q_lo = ((sbase + Ly::kQOff) >> 4) | (1u << 16);
      const uint32_t k_lo = ((sbase + Ly::kKOff) >> 4) | (1u << 16);
      // V is MN-major: LBO = one box (the two 64-column halves of dv)
      const uint32_t v_lo = ((sbase + Ly::kVOff) >> 4) | ((Ly::kKBox >> 4) << 16);
      uint32_t gi = 0, gk = 0, gv = 0, gp = 0;
      bool ok = true, issued = false;
      auto qk = [&](int32_t x, uint32_t st) {
        const uint32_t a_lo = q_lo + x * (kQStageBytes >> 4);
        const uint32_t b_lo = k_lo + st * (Ly::kKStage >> 4);
#pragma unroll
        for (int kstep = 0; kstep < kDqk / 16; ++kstep) {
          const uint32_t box = kstep >> 2, off = (kstep & 3) * 32;
          mma_ss2(tmem + x * 128, a_lo + ((box * kQBoxBytes + off) >> 4), kDescHi,
                  b_lo + ((box * Ly::kKBox + off) >> 4), kDescHi, box == 0 ? kIdQKRot : kIdQK,
                  kstep > 0 ? 1u : 0u);
        }
        mma_commit(B_SFULL(x));
      };
      auto pv = [&](int32_t x, bool first) -> bool {
        if (!wait_bar(B_PFULL(x), gp & 1, abort_flag, 4)) return false;
        tc_fence_after();
        if (first) {
          if (!wait_bar(B_OEMPTY(x), (gi & 1) ^ 1, abort_flag, 5)) return false;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < kCauBN / 16; ++kk)
          mma_ts2(tmem + 256 + x * 128, tmem + x * 128 + kk * 8, v_lo + kk * 128, kDescHi, kIdPV,
                  (!first || kk > 0) ? 1u : 0u);
        mma_commit(B_PVDONE(x));
        return true;
      };
      auto kready = [&](uint32_t g) {
        return wait_bar(B_KREADY(g & 1), (g >> 1) & 1, abort_flag, 6);
      };
      for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
        const CauItem it = cau_item(args, w);
        if (!it.valid) continue;
        if (!(ok = wait_bar(B_QREADY(0), gi & 1, abort_flag, 3) &&
                   wait_bar(B_QREADY(1), gi & 1, abort_flag, 3)))
          break;
        if (!(ok = kready(gk))) break;
        tc_fence_after();
        qk(0, gk & 1);
        qk(1, gk & 1);
        issued = true;
        mma_commit(B_KEMPTY(gk & 1));
        if (it.nblk == 1) mma_commit(B_QEMPTY);
        for (int32_t j = 0; ok && j < it.nblk; ++j) {
          const bool more = j + 1 < it.nblk;
          if (!(ok = wait_bar(B_VFULL, gv & 1, abort_flag, 13))) break;
          tc_fence_after();
          if (!(ok = pv(0, j == 0))) break;
          if (more) {
            if (!(ok = kready(gk + 1))) break;
            tc_fence_after();
            qk(0, (gk + 1) & 1);
          }
          if (!(ok = pv(1, j == 0))) break;
          mma_commit(B_VEMPTY);
          ++gv;
          ++gp;
          if (more) {
            qk(1, (gk + 1) & 1);
            mma_commit(B_KEMPTY((gk + 1) & 1));
            if (j + 1 == it.nblk - 1) mma_commit(B_QEMPTY);
          }
          ++gk;
        }
        ++gi;
      }
      if (issued) {
        mma_commit(B_DRAIN);
        drain_wait(B_DRAIN, 0);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ============================================================ softmax + epilogue
    cau_softmax(args, warp < 8 ? 0 : 1, tmem, sbase, abort_flag);
  } else if (warp >= 12) {
    // ============================================================ RoPE
    const int32_t tid = threadIdx.x - 384;
    uint32_t gi = 0, gk = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; ok && w < args.n_items; w += gridDim.x) {
      const CauItem it = cau_item(args, w);
      if (!it.valid) continue;
      for (int32_t x = 0; ok && x < 2; ++x) {
        if (!(ok = wait_bar_warp(B_QFULL(x), gi & 1, abort_flag, 10))) break;
        const int32_t p0 = it.t0 + x * args.T;
        const int32_t ntok = min(args.T, it.L - p0);  // tile B may lie past the end
        if (args.rope_on && ntok > 0)
          rope_q_tile(smem + Ly::kQOff + x * kQStageBytes, G, ntok, p0, args.rope_style, turns, tid);
        fence_proxy_async_smem();
        mbar_arrive(B_QREADY(x));
      }
      if (!ok) break;
      ++gi;
      for (int32_t j = 0; j < it.nblk; ++j) {
        const uint32_t st = gk & 1;
        if (!(ok = wait_bar_warp(B_KFULL(st), (gk >> 1) & 1, abort_flag, 11))) break;
        if (args.rope_on)
          rope_k_rows(smem + Ly::kKOff + st * Ly::kKStage, kCauBN, (it.kb0 + j) * kCauBN,
                      args.rope_style, turns, tid);
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
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace sa
