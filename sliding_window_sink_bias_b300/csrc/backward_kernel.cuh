// backward_kernel.cuh -- backward pass of the sink-bias GQA attention prefill.
//
// The MiMo-V2-Flash Technical Report trains the sink logits (§2.2: one
// learnable sink per head); its eqs. (1)-(3) define the forward only, and the
// backward here is the plain chain rule through them, for L = sum dO . o:
//   s_ij = exp(a_ij - lse_i)            (lse from the forward, sink included)
//   D_i = dO_i . o_i,  dP_ij = dO_i . v_j,  dS_ij = s_ij (dP_ij - D_i)
//   dv_j = sum_i s_ij dO_i
//   dq~_i = scale sum_j dS_ij k~_j,  dk~_j = scale sum_i dS_ij q~_i  (rotated q~, k~)
//   dsink_h = -sum_i exp(sink_h - lse_i) D_i
// and dq, dk are the gradients turned back by the transposed rotation.
//
// Four launches:
//   bwd_pre_kernel    per token: D_i for every head, RoPE-rotated copies of q
//                     and k (bf16, workspace), and per-chunk partial sums of
//                     the sink gradient (fixed order: the result is the same
//                     bits every run).
//   bwd_dq_kernel     per tile of 128 packed query rows (G heads x 128/G tokens
//                     of one KV head), over 64-key blocks: S = Q K^T and
//                     dP = dO V^T on tcgen05 into TMEM, dS in registers, back to
//                     TMEM as bf16, dQ += dS K (A from TMEM); epilogue dQ * scale,
//                     inverse RoPE, bf16.
//   bwd_dkdv_kernel   per block of 128 keys of one KV head, over sub-tiles of 64
//                     packed query rows: S^T = K Q^T and dP^T = V dO^T into TMEM,
//                     P^T and dS^T in registers, back to TMEM as bf16,
//                     dV += P^T dO and dK += dS^T Q (A from TMEM, B = the same
//                     shared-memory tiles read N-major); epilogue as above.
//   bwd_dsink_kernel  the per-chunk partials summed in chunk order.
//
// The MMA kernels are synchronous (one batch of MMAs in flight; the next K/V
// block or Q sub-tile is prefetched by TMA while the current one is worked
// on), 128 threads, one row per thread (TMEM lane); every wait is bounded and
// every CTA-wide decision is taken with __syncthreads_and.
#pragma once
#include "common.cuh"

namespace sa {

constexpr int32_t kBwdThreads = 128;
constexpr int32_t kBwdChunk = 32;    // tokens per pre-pass CTA
constexpr int32_t kDqBN = 64;        // keys per block (dq kernel)
constexpr int32_t kKvBN = 128;       // keys per block (dkdv kernel)
constexpr int32_t kKvRows = 64;      // packed query rows per sub-tile (dkdv kernel)

struct BwdArgs {
  int32_t Hq, Hkv, G;
  int32_t batch, total;
  int32_t window;
  int32_t rope_on, rope_style;
  float scale, scale_log2;
  const int32_t *cu_seqlens;
  const float *sink;
  const __nv_bfloat16 *q, *k, *out, *dout;
  const float *lse;
  __nv_bfloat16 *q_rot, *k_rot;
  float *D, *dsink_part;
  int32_t n_chunks;
  __nv_bfloat16 *dq, *dk, *dv;
  float *dsink;
  int32_t dq_tiles, dq_items;   // tiles per sequence (virtual, of 128/G tokens), items
  int32_t kv_blocks, kv_items;  // key blocks per sequence (virtual), items
  unsigned long long rope_turns[32];
};

// Sequence of a token (binary search over cu_seqlens).
__device__ __forceinline__ int32_t bwd_seq_of(const BwdArgs &a, int32_t tok) {
  int32_t lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (__ldg(a.cu_seqlens + mid) <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------------ pre-pass
// One warp per token (chunk of kBwdChunk tokens per CTA, 256 threads).  Lane l
// owns rotary pair l (dims (2l, 2l+1) or (l, l+32)) and dims 64+4l..64+4l+3.
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __grid_constant__ BwdArgs a) {
  __shared__ float sD[kBwdChunk][64];  // D of the chunk's tokens (heads < 64 cached here)
  const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t tok0 = blockIdx.x * kBwdChunk;
  for (int32_t tt = warp; tt < kBwdChunk; tt += 8) {
    const int32_t tok = tok0 + tt;
    if (tok >= a.total) break;
    const int32_t b = bwd_seq_of(a, tok);
    const int32_t pos = tok - __ldg(a.cu_seqlens + b);
    float c = 1.f, s = 0.f;
    if (a.rope_on) rope_cs(pos, a.rope_turns[lane], c, s);
    const int32_t ia = a.rope_style == 0 ? 2 * lane : lane;
    const int32_t ib = a.rope_style == 0 ? 2 * lane + 1 : lane + 32;
    // rotated copies: q (Hq heads) then k (Hkv heads)
    for (int32_t hh = 0; hh < a.Hq + a.Hkv; ++hh) {
      const bool isq = hh < a.Hq;
      const size_t row = isq ? static_cast<size_t>(tok) * a.Hq + hh
                             : static_cast<size_t>(tok) * a.Hkv + (hh - a.Hq);
      const __nv_bfloat16 *src = (isq ? a.q : a.k) + row * kDqk;
      __nv_bfloat16 *dst = (isq ? a.q_rot : a.k_rot) + row * kDqk;
      const float x = __bfloat162float(src[ia]), y = __bfloat162float(src[ib]);
      dst[ia] = __float2bfloat16_rn(x * c - y * s);
      dst[ib] = __float2bfloat16_rn(x * s + y * c);
      *reinterpret_cast<uint2 *>(dst + 64 + 4 * lane) =
          *reinterpret_cast<const uint2 *>(src + 64 + 4 * lane);
    }
    // D = dO . o per head (4 dims per lane, warp sum)
    for (int32_t h = 0; h < a.Hq; ++h) {
      const size_t row = static_cast<size_t>(tok) * a.Hq + h;
      const uint2 ov = *reinterpret_cast<const uint2 *>(a.out + row * kDv + 4 * lane);
      const uint2 dv = *reinterpret_cast<const uint2 *>(a.dout + row * kDv + 4 * lane);
      float acc = bf16lo(ov.x) * bf16lo(dv.x) + bf16hi(ov.x) * bf16hi(dv.x) +
                  bf16lo(ov.y) * bf16lo(dv.y) + bf16hi(ov.y) * bf16hi(dv.y);
#pragma unroll
      for (int32_t o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) {
        a.D[row] = acc;
        if (h < 64) sD[tt][h] = acc;
      }
    }
  }
  __syncthreads();
  // partial sink gradient of this chunk, per head, tokens in order
  for (int32_t h = threadIdx.x; h < a.Hq; h += blockDim.x) {
    const float sk = __ldg(a.sink + h);
    float acc = 0.f;
    if (sk != -INFINITY) {
      for (int32_t tt = 0; tt < kBwdChunk; ++tt) {
        const int32_t tok = tok0 + tt;
        if (tok >= a.total) break;
        const size_t row = static_cast<size_t>(tok) * a.Hq + h;
        const float l = __ldg(a.lse + row);
        const float d = h < 64 ? sD[tt][h] : a.D[row];
        if (l != -INFINITY) acc -= ex2((sk - l) * kLog2e) * d;
      }
    }
    a.dsink_part[static_cast<size_t>(blockIdx.x) * a.Hq + h] = acc;
  }
}

__global__ void __launch_bounds__(256) bwd_dsink_kernel(const __grid_constant__ BwdArgs a) {
  for (int32_t h = threadIdx.x; h < a.Hq; h += blockDim.x) {
    float acc = 0.f;
    for (int32_t c = 0; c < a.n_chunks; ++c) acc += a.dsink_part[static_cast<size_t>(c) * a.Hq + h];
    a.dsink[h] = acc;
  }
}

// ------------------------------------------------------------------ shared pieces
// TMEM columns: S (or S^T) 0..63, dP (or dP^T) 64..127, accumulators from 128.
constexpr uint32_t kBwdColS = 0, kBwdColP = 64, kBwdColAcc = 128;
constexpr uint32_t kBwdDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);  // SW128, SBO 1024

// Inverse RoPE on dims 0..63 held in x[64] (fp32), at position pos.
__device__ __forceinline__ void bwd_unrotate(float (&x)[64], int32_t pos, int32_t style,
                                             const unsigned long long *turns) {
  // the pairing is a compile-time index pattern in each branch, so x stays in registers
  if (style == 0) {
#pragma unroll
    for (int32_t t = 0; t < 32; ++t) {
      float c, s;
      rope_cs(pos, turns[t], c, s);
      const float u = x[2 * t], w = x[2 * t + 1];
      x[2 * t] = u * c + w * s;
      x[2 * t + 1] = w * c - u * s;
    }
  } else {
#pragma unroll
    for (int32_t t = 0; t < 32; ++t) {
      float c, s;
      rope_cs(pos, turns[t], c, s);
      const float u = x[t], w = x[t + 32];
      x[t] = u * c + w * s;
      x[t + 32] = w * c - u * s;
    }
  }
}

// Row epilogue shared by the gradients of q and k: 192 fp32 columns of TMEM at
// col (this thread's lane) -> * scale, inverse RoPE on dims 0..63, bf16 row.
__device__ __forceinline__ void bwd_store_qk_row(uint32_t t_col, float scale, bool rope_on,
                                                 int32_t style, int32_t pos,
                                                 const unsigned long long *turns,
                                                 __nv_bfloat16 *dst, bool valid) {
  {
    uint32_t r[64];
    tmem_ld32p(t_col, r);
    tmem_ld32p(t_col + 32, r + 32);
    tmem_wait_ld();
    reg_fence<64>(r);
    float x[64];
#pragma unroll
    for (int32_t e = 0; e < 64; ++e) x[e] = __uint_as_float(r[e]) * scale;
    if (rope_on) bwd_unrotate(x, pos, style, turns);
    if (valid) {
#pragma unroll
      for (int32_t e = 0; e < 64; e += 8) {
        *reinterpret_cast<uint4 *>(dst + e) =
            make_uint4(pack_bf16x2(x[e], x[e + 1]), pack_bf16x2(x[e + 2], x[e + 3]),
                       pack_bf16x2(x[e + 4], x[e + 5]), pack_bf16x2(x[e + 6], x[e + 7]));
      }
    }
  }
#pragma unroll 1
  for (int32_t cb = 64; cb < 192; cb += 32) {
    uint32_t r[32];
    tmem_ld32p(t_col + cb, r);
    tmem_wait_ld();
    reg_fence<32>(r);
    if (valid) {
#pragma unroll
      for (int32_t e = 0; e < 32; e += 8) {
        const float *f = reinterpret_cast<const float *>(r + e);
        *reinterpret_cast<uint4 *>(dst + cb + e) =
            make_uint4(pack_bf16x2(f[0] * scale, f[1] * scale), pack_bf16x2(f[2] * scale, f[3] * scale),
                       pack_bf16x2(f[4] * scale, f[5] * scale), pack_bf16x2(f[6] * scale, f[7] * scale));
      }
    }
  }
}

// ------------------------------------------------------------------ dQ kernel
struct DqLayout {
  static constexpr uint32_t kQBox = 128 * kRowBytes;     // 128 rows x 64 dims: 16 KB
  static constexpr uint32_t kKBox = kDqBN * kRowBytes;   // 64 keys x 64 dims: 8 KB
  static constexpr uint32_t kQOff = 0;                   // q_rot tile: 3 boxes
  static constexpr uint32_t kDoOff = 3 * kQBox;          // dO tile: 2 boxes
  static constexpr uint32_t kStOff = 5 * kQBox;          // stages: K 3 boxes, V 2 boxes
  static constexpr uint32_t kStage = 5 * kKBox;
  static constexpr uint32_t kBarOff = kStOff + 2 * kStage;  // qf, kv[2], mm1, mm2
  static constexpr uint32_t kMiscOff = kBarOff + 5 * 8;      // tmem slot, abort flag
  static constexpr uint32_t kBytes = kMiscOff + 16;
  static constexpr uint32_t kDynSmem = kBytes + 1024;
};
static_assert(DqLayout::kDynSmem <= 232448, "dq kernel shared memory");

__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ BwdArgs a) {
  using Ly = DqLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int32_t warp = threadIdx.x >> 5;
  const int32_t row = threadIdx.x;  // packed query row == TMEM lane
  const bool issuer = threadIdx.x == 0;
  const uint32_t B_QF = sbase + Ly::kBarOff, B_MM1 = B_QF + 24, B_MM2 = B_QF + 32;
  auto B_KV = [&](uint32_t s) { return B_QF + 8 + 8 * s; };
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  if (issuer) {
    mbar_init(B_QF, 1);
    mbar_init(B_KV(0), 1);
    mbar_init(B_KV(1), 1);
    mbar_init(B_MM1, 1);
    mbar_init(B_MM2, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(sbase + Ly::kMiscOff, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_t = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int32_t G = a.G, T = 128 / G;
  const int32_t t_row = row / G, g_row = row % G;
  const uint32_t q_lo = ((sbase + Ly::kQOff) >> 4) | (1u << 16);
  const uint32_t do_lo = ((sbase + Ly::kDoOff) >> 4) | (1u << 16);
  constexpr uint32_t kIdS = idesc_f32acc(128, kDqBN, 1, 0, 0);
  constexpr uint32_t kIdQ = idesc_f32acc(128, kDqk, 1, 0, 1);
  uint32_t n_qf = 0, n_kv[2] = {0, 0}, n_m1 = 0, n_m2 = 0, gk = 0;
  bool ok = true;
  for (int32_t it = blockIdx.x; ok && it < a.dq_items; it += gridDim.x) {
    // item -> (sequence, KV head, tile); global tiles longest first
    const int32_t per_seq = a.Hkv * a.dq_tiles;
    const int32_t b = it / per_seq, rem = it % per_seq;
    const int32_t kvh = rem % a.Hkv;
    const int32_t tile = a.window > 0 ? rem / a.Hkv : a.dq_tiles - 1 - rem / a.Hkv;
    const int32_t s0 = __ldg(a.cu_seqlens + b), L = __ldg(a.cu_seqlens + b + 1) - s0;
    const int32_t t0 = tile * T;
    if (t0 >= L) continue;
    const int32_t lo = a.window > 0 ? max(0, t0 - a.window + 1) : 0;
    const int32_t hi = min(L, t0 + T) - 1;
    const int32_t nblk = (hi - lo + kDqBN) / kDqBN;
    // this thread's row
    const int32_t ti = t0 + t_row, h = kvh * G + g_row;
    const bool rvalid = ti < L;
    const size_t grow = static_cast<size_t>(s0 + ti) * a.Hq + h;
    const float lse2 = rvalid ? __ldg(a.lse + grow) * kLog2e : 0.f;
    const float Drow = rvalid ? __ldg(a.D + grow) : 0.f;
    if (issuer) {
      mbar_arrive_expect_tx(B_QF, 5 * Ly::kQBox);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc)
        tma_load_3d(sbase + Ly::kQOff + cc * Ly::kQBox, &tm_q, cc * 64, kvh * G, s0 + t0, B_QF);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(sbase + Ly::kDoOff + cc * Ly::kQBox, &tm_do, cc * 64, kvh * G, s0 + t0, B_QF);
    }
    ++n_qf;
    auto load_block = [&](int32_t j, uint32_t st) {
      const uint32_t dst = sbase + Ly::kStOff + st * Ly::kStage;
      const int32_t krow = s0 + lo + j * kDqBN;
      mbar_arrive_expect_tx(B_KV(st), Ly::kStage);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc) tma_load_3d(dst + cc * Ly::kKBox, &tm_k, cc * 64, kvh, krow, B_KV(st));
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(dst + (3 + cc) * Ly::kKBox, &tm_v, cc * 64, kvh, krow, B_KV(st));
    };
    if (issuer) load_block(0, gk & 1);
    ++n_kv[gk & 1];
    ok = wait_bar(B_QF, (n_qf - 1) & 1, abort_flag, 20);
    ok = __syncthreads_and(ok);
    for (int32_t j = 0; ok && j < nblk; ++j, ++gk) {
      const uint32_t st = gk & 1;
      if (j + 1 < nblk) {
        if (issuer) load_block(j + 1, st ^ 1);
        ++n_kv[st ^ 1];
      }
      ok = wait_bar(B_KV(st), (n_kv[st] - 1) & 1, abort_flag, 21);
      ok = __syncthreads_and(ok);
      if (!ok) break;
      const uint32_t k_lo = ((sbase + Ly::kStOff + st * Ly::kStage) >> 4) | (1u << 16);
      const uint32_t v_lo = k_lo + ((3 * Ly::kKBox) >> 4);
      if (issuer) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kDqk / 16; ++ks) {
          const uint32_t ao = ((ks >> 2) * Ly::kQBox + (ks & 3) * 32) >> 4;
          const uint32_t bo = ((ks >> 2) * Ly::kKBox + (ks & 3) * 32) >> 4;
          mma_ss2(tmem + kBwdColS, q_lo + ao, kBwdDescHi, k_lo + bo, kBwdDescHi, kIdS, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < kDv / 16; ++ks) {
          const uint32_t ao = ((ks >> 2) * Ly::kQBox + (ks & 3) * 32) >> 4;
          const uint32_t bo = ((ks >> 2) * Ly::kKBox + (ks & 3) * 32) >> 4;
          mma_ss2(tmem + kBwdColP, do_lo + ao, kBwdDescHi, v_lo + bo, kBwdDescHi, kIdS, ks > 0);
        }
        mma_commit(B_MM1);
      }
      ++n_m1;
      ok = wait_bar(B_MM1, (n_m1 - 1) & 1, abort_flag, 22);
      ok = __syncthreads_and(ok);
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t sv[64], pv[64];
        tmem_ld32p(lane_t + kBwdColS, sv);
        tmem_ld32p(lane_t + kBwdColS + 32, sv + 32);
        tmem_ld32p(lane_t + kBwdColP, pv);
        tmem_ld32p(lane_t + kBwdColP + 32, pv + 32);
        tmem_wait_ld();
        reg_fence<64>(sv);
        reg_fence<64>(pv);
        const int32_t kb = lo + j * kDqBN;
#pragma unroll
        for (int32_t c = 0; c < kDqBN; c += 2) {
          float ds[2];
#pragma unroll
          for (int32_t e = 0; e < 2; ++e) {
            const int32_t kj = kb + c + e;
            const bool vis = rvalid && kj <= ti && (a.window == 0 || kj > ti - a.window);
            const float p = vis ? ex2(__uint_as_float(sv[c + e]) * a.scale_log2 - lse2) : 0.f;
            ds[e] = p * (__uint_as_float(pv[c + e]) - Drow);
          }
          sv[c >> 1] = pack_bf16x2(ds[0], ds[1]);
        }
        tmem_st32p(lane_t + kBwdColS, sv);  // dS as bf16 pairs over S
        tmem_wait_st();
      }
      tc_fence_before();
      ok = __syncthreads_and(ok);
      if (!ok) break;
      if (issuer) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kDqBN / 16; ++ks)
          mma_ts2(tmem + kBwdColAcc, tmem + kBwdColS + ks * 8,
                  ((sbase + Ly::kStOff + st * Ly::kStage) >> 4) + ks * ((16 * kRowBytes) >> 4) +
                      ((Ly::kKBox >> 4) << 16),
                  kBwdDescHi, kIdQ, (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(B_MM2);
      }
      ++n_m2;
      ok = wait_bar(B_MM2, (n_m2 - 1) & 1, abort_flag, 23);
      ok = __syncthreads_and(ok);
    }
    if (!ok) break;
    tc_fence_after();
    bwd_store_qk_row(lane_t + kBwdColAcc, a.scale, a.rope_on, a.rope_style, ti, a.rope_turns,
                     a.dq + grow * kDqk, rvalid);
    tc_fence_before();
    ok = __syncthreads_and(ok);
  }
  // drain: every copy and MMA this CTA issued must land before TMEM and shared
  // memory go back (only an aborted CTA has any left)
  if (n_qf > 0) drain_wait(B_QF, (n_qf - 1) & 1);
  for (uint32_t s = 0; s < 2; ++s)
    if (n_kv[s] > 0) drain_wait(B_KV(s), (n_kv[s] - 1) & 1);
  if (n_m1 > 0) drain_wait(B_MM1, (n_m1 - 1) & 1);
  if (n_m2 > 0) drain_wait(B_MM2, (n_m2 - 1) & 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dK / dV kernel
struct KvLayout {
  static constexpr uint32_t kKBox = kKvBN * kRowBytes;   // 128 keys x 64 dims: 16 KB
  static constexpr uint32_t kQBox = kKvRows * kRowBytes; // 64 rows x 64 dims: 8 KB
  static constexpr uint32_t kKOff = 0;                   // k_rot block: 3 boxes
  static constexpr uint32_t kVOff = 3 * kKBox;           // v block: 2 boxes
  static constexpr uint32_t kStOff = 5 * kKBox;          // stages: q_rot rows 3 boxes, dO rows 2
  static constexpr uint32_t kStage = 5 * kQBox;
  static constexpr uint32_t kColOff = kStOff + 2 * kStage;  // lse*log2e, D of the sub-tile's rows
  static constexpr uint32_t kBarOff = kColOff + 2 * kKvRows * 4;  // kf, qs[2], mm1, mm2
  static constexpr uint32_t kMiscOff = kBarOff + 5 * 8;
  static constexpr uint32_t kBytes = kMiscOff + 16;
  static constexpr uint32_t kDynSmem = kBytes + 1024;
};
static_assert(KvLayout::kDynSmem <= 232448, "dkdv kernel shared memory");

__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ BwdArgs a) {
  using Ly = KvLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int32_t warp = threadIdx.x >> 5;
  const int32_t lane_row = threadIdx.x;  // key row == TMEM lane
  const bool issuer = threadIdx.x == 0;
  const uint32_t B_KF = sbase + Ly::kBarOff, B_MM1 = B_KF + 24, B_MM2 = B_KF + 32;
  auto B_QS = [&](uint32_t s) { return B_KF + 8 + 8 * s; };
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  float *c_lse = reinterpret_cast<float *>(smem + Ly::kColOff);
  float *c_D = c_lse + kKvRows;
  if (issuer) {
    mbar_init(B_KF, 1);
    mbar_init(B_QS(0), 1);
    mbar_init(B_QS(1), 1);
    mbar_init(B_MM1, 1);
    mbar_init(B_MM2, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(sbase + Ly::kMiscOff, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_t = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int32_t G = a.G, TS = kKvRows / G;  // tokens per sub-tile
  const uint32_t k_lo = ((sbase + Ly::kKOff) >> 4) | (1u << 16);
  const uint32_t v_lo = ((sbase + Ly::kVOff) >> 4) | (1u << 16);
  constexpr uint32_t kIdS = idesc_f32acc(128, kKvRows, 1, 0, 0);
  constexpr uint32_t kIdV = idesc_f32acc(128, kDv, 1, 0, 1);
  constexpr uint32_t kIdK = idesc_f32acc(128, kDqk, 1, 0, 1);
  constexpr uint32_t kColV = kBwdColAcc, kColK = kBwdColAcc + kDv;  // 128..255, 256..447
  uint32_t n_kf = 0, n_qs[2] = {0, 0}, n_m1 = 0, n_m2 = 0, gs = 0;
  bool ok = true;
  for (int32_t it = blockIdx.x; ok && it < a.kv_items; it += gridDim.x) {
    const int32_t per_seq = a.Hkv * a.kv_blocks;
    const int32_t b = it / per_seq, rem = it % per_seq;
    const int32_t kvh = rem % a.Hkv;
    const int32_t blk = rem / a.Hkv;  // global: the earliest blocks (most queries) first
    const int32_t s0 = __ldg(a.cu_seqlens + b), L = __ldg(a.cu_seqlens + b + 1) - s0;
    const int32_t k0 = blk * kKvBN;
    if (k0 >= L) continue;
    const int32_t i_lo = k0;
    const int32_t i_hi = a.window > 0 ? min(L - 1, k0 + kKvBN - 1 + a.window - 1) : L - 1;
    const int32_t nsub = (i_hi - i_lo + TS) / TS;
    const int32_t kj = k0 + lane_row;  // this thread's key
    const bool kvalid = kj < L;
    if (issuer) {
      mbar_arrive_expect_tx(B_KF, 5 * Ly::kKBox);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc)
        tma_load_3d(sbase + Ly::kKOff + cc * Ly::kKBox, &tm_k, cc * 64, kvh, s0 + k0, B_KF);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(sbase + Ly::kVOff + cc * Ly::kKBox, &tm_v, cc * 64, kvh, s0 + k0, B_KF);
    }
    ++n_kf;
    auto load_sub = [&](int32_t sidx, uint32_t st) {
      const uint32_t dst = sbase + Ly::kStOff + st * Ly::kStage;
      const int32_t tok = s0 + i_lo + sidx * TS;
      mbar_arrive_expect_tx(B_QS(st), Ly::kStage);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc) tma_load_3d(dst + cc * Ly::kQBox, &tm_q, cc * 64, kvh * G, tok, B_QS(st));
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(dst + (3 + cc) * Ly::kQBox, &tm_do, cc * 64, kvh * G, tok, B_QS(st));
    };
    if (issuer) load_sub(0, gs & 1);
    ++n_qs[gs & 1];
    ok = wait_bar(B_KF, (n_kf - 1) & 1, abort_flag, 24);
    ok = __syncthreads_and(ok);
    for (int32_t sidx = 0; ok && sidx < nsub; ++sidx, ++gs) {
      const uint32_t st = gs & 1;
      if (sidx + 1 < nsub) {
        if (issuer) load_sub(sidx + 1, st ^ 1);
        ++n_qs[st ^ 1];
      }
      const int32_t i0 = i_lo + sidx * TS;
      if (threadIdx.x < kKvRows) {
        const int32_t ti = i0 + threadIdx.x / G, h = kvh * G + threadIdx.x % G;
        const bool v = ti < L;
        const size_t grow = static_cast<size_t>(s0 + ti) * a.Hq + h;
        c_lse[threadIdx.x] = v ? __ldg(a.lse + grow) * kLog2e : 0.f;
        c_D[threadIdx.x] = v ? __ldg(a.D + grow) : 0.f;
      }
      ok = wait_bar(B_QS(st), (n_qs[st] - 1) & 1, abort_flag, 25);
      ok = __syncthreads_and(ok);
      if (!ok) break;
      const uint32_t q_lo = ((sbase + Ly::kStOff + st * Ly::kStage) >> 4) | (1u << 16);
      const uint32_t do_lo = q_lo + ((3 * Ly::kQBox) >> 4);
      if (issuer) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kDqk / 16; ++ks) {
          const uint32_t ao = ((ks >> 2) * Ly::kKBox + (ks & 3) * 32) >> 4;
          const uint32_t bo = ((ks >> 2) * Ly::kQBox + (ks & 3) * 32) >> 4;
          mma_ss2(tmem + kBwdColS, k_lo + ao, kBwdDescHi, q_lo + bo, kBwdDescHi, kIdS, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < kDv / 16; ++ks) {
          const uint32_t ao = ((ks >> 2) * Ly::kKBox + (ks & 3) * 32) >> 4;
          const uint32_t bo = ((ks >> 2) * Ly::kQBox + (ks & 3) * 32) >> 4;
          mma_ss2(tmem + kBwdColP, v_lo + ao, kBwdDescHi, do_lo + bo, kBwdDescHi, kIdS, ks > 0);
        }
        mma_commit(B_MM1);
      }
      ++n_m1;
      ok = wait_bar(B_MM1, (n_m1 - 1) & 1, abort_flag, 26);
      ok = __syncthreads_and(ok);
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t sv[64], pv[64];
        tmem_ld32p(lane_t + kBwdColS, sv);
        tmem_ld32p(lane_t + kBwdColS + 32, sv + 32);
        tmem_ld32p(lane_t + kBwdColP, pv);
        tmem_ld32p(lane_t + kBwdColP + 32, pv + 32);
        tmem_wait_ld();
        reg_fence<64>(sv);
        reg_fence<64>(pv);
#pragma unroll
        for (int32_t c = 0; c < kKvRows; c += 2) {
          float pp[2], ds[2];
#pragma unroll
          for (int32_t e = 0; e < 2; ++e) {
            const int32_t ti = i0 + (c + e) / G;
            const bool vis = kvalid && ti < L && kj <= ti && (a.window == 0 || kj > ti - a.window);
            pp[e] = vis ? ex2(__uint_as_float(sv[c + e]) * a.scale_log2 - c_lse[c + e]) : 0.f;
            ds[e] = pp[e] * (__uint_as_float(pv[c + e]) - c_D[c + e]);
          }
          sv[c >> 1] = pack_bf16x2(pp[0], pp[1]);
          pv[c >> 1] = pack_bf16x2(ds[0], ds[1]);
        }
        tmem_st32p(lane_t + kBwdColS, sv);  // P^T as bf16 pairs over S^T
        tmem_st32p(lane_t + kBwdColP, pv);  // dS^T as bf16 pairs over dP^T
        tmem_wait_st();
      }
      tc_fence_before();
      ok = __syncthreads_and(ok);
      if (!ok) break;
      if (issuer) {
        tc_fence_after();
        const uint32_t stb = (sbase + Ly::kStOff + st * Ly::kStage) >> 4;
#pragma unroll
        for (int ks = 0; ks < kKvRows / 16; ++ks) {
          const uint32_t step = ks * ((16 * kRowBytes) >> 4);
          // dV += P^T dO: B = the dO rows read N-major (LBO = one box)
          mma_ts2(tmem + kColV, tmem + kBwdColS + ks * 8,
                  stb + ((3 * Ly::kQBox) >> 4) + step + ((Ly::kQBox >> 4) << 16), kBwdDescHi, kIdV,
                  (sidx > 0 || ks > 0) ? 1u : 0u);
          // dK += dS^T Q: B = the q_rot rows read N-major
          mma_ts2(tmem + kColK, tmem + kBwdColP + ks * 8, stb + step + ((Ly::kQBox >> 4) << 16),
                  kBwdDescHi, kIdK, (sidx > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(B_MM2);
      }
      ++n_m2;
      ok = wait_bar(B_MM2, (n_m2 - 1) & 1, abort_flag, 27);
      ok = __syncthreads_and(ok);
    }
    if (!ok) break;
    tc_fence_after();
    {
      // dV row: 128 fp32 columns -> bf16
      __nv_bfloat16 *dst = a.dv + (static_cast<size_t>(s0 + kj) * a.Hkv + kvh) * kDv;
#pragma unroll 1
      for (int32_t cb = 0; cb < kDv; cb += 32) {
        uint32_t r[32];
        tmem_ld32p(lane_t + kColV + cb, r);
        tmem_wait_ld();
        reg_fence<32>(r);
        if (kvalid) {
#pragma unroll
          for (int32_t e = 0; e < 32; e += 8) {
            const float *f = reinterpret_cast<const float *>(r + e);
            *reinterpret_cast<uint4 *>(dst + cb + e) =
                make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                           pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
          }
        }
      }
    }
    bwd_store_qk_row(lane_t + kColK, a.scale, a.rope_on, a.rope_style, kj, a.rope_turns,
                     a.dk + (static_cast<size_t>(s0 + kj) * a.Hkv + kvh) * kDqk, kvalid);
    tc_fence_before();
    ok = __syncthreads_and(ok);
  }
  if (n_kf > 0) drain_wait(B_KF, (n_kf - 1) & 1);
  for (uint32_t s = 0; s < 2; ++s)
    if (n_qs[s] > 0) drain_wait(B_QS(s), (n_qs[s] - 1) & 1);
  if (n_m1 > 0) drain_wait(B_MM1, (n_m1 - 1) & 1);
  if (n_m2 > 0) drain_wait(B_MM2, (n_m2 - 1) & 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace sa
