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
//   bwd_dsink_kernel  the per-chunk partials summed in a fixed order, one CTA
//                     per head.
//
// The MMA kernels run 8 warps that own half a row each (TMEM lane; warps w and
// w + 4 share the lanes of w % 4), a ninth warp whose first thread issues the
// MMAs and a tenth whose first thread issues the copies, so neither the rows
// nor the MMAs wait for the other issuing; every wait is bounded and every
// CTA-wide decision is taken with __syncthreads_and.
#pragma once
#include "common.cuh"

namespace sa {

constexpr int32_t kBwdThreads = 320;  // dq / dkdv: 8 row warps, an MMA warp, a copy warp
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
  __nv_bfloat16 *q_rot, *k_rot;  // rotated dims 0..63: [total, Hq, 64], [total, Hkv, 64]
  float *D, *dsink_part;
  int32_t n_chunks;
  __nv_bfloat16 *dq, *dk, *dv;
  float *dsink;
  int32_t dq_tiles, dq_items;   // tiles per sequence (virtual, of 128/G tokens), items
  int32_t kv_blocks, kv_items;  // key blocks per sequence (virtual), items
  int32_t grad_v8;              // dq, dk, dv 32-byte aligned (whole-sector stores)
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
// owns rotary pair l (dims (2l, 2l+1) or (l, l+32)).  Only the 64 rotated dims
// of q and k are written out (the MMA kernels read dims 64..191 from q and k
// themselves); without RoPE nothing is.
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __grid_constant__ BwdArgs a) {
  __shared__ float sD[kBwdChunk][64];  // D of the chunk's tokens (heads < 64 cached here)
  const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t tok0 = blockIdx.x * kBwdChunk;
  for (int32_t tt = warp; tt < kBwdChunk; tt += 8) {
    const int32_t tok = tok0 + tt;
    if (tok >= a.total) break;
    const int32_t b = bwd_seq_of(a, tok);
    const int32_t pos = tok - __ldg(a.cu_seqlens + b);
    if (a.rope_on && a.rope_style == 0) {
      float c, s;
      rope_cs(pos, a.rope_turns[lane], c, s);
      // rotated rows: q (Hq heads) then k (Hkv heads), in 16-byte units (8 a
      // row).  Pairs (2t, 2t+1): unit c of a row holds pairs 4c..4c+3, whose
      // angles lanes 4c..4c+3 computed above; lane l works on unit l % 8, so
      // it fetches the same four angles in every round.
      const int32_t cc = lane & 7;
      const float c0 = __shfl_sync(0xffffffffu, c, 4 * cc), s0 = __shfl_sync(0xffffffffu, s, 4 * cc);
      const float c1 = __shfl_sync(0xffffffffu, c, 4 * cc + 1), s1 = __shfl_sync(0xffffffffu, s, 4 * cc + 1);
      const float c2 = __shfl_sync(0xffffffffu, c, 4 * cc + 2), s2 = __shfl_sync(0xffffffffu, s, 4 * cc + 2);
      const float c3 = __shfl_sync(0xffffffffu, c, 4 * cc + 3), s3 = __shfl_sync(0xffffffffu, s, 4 * cc + 3);
      const int32_t nunit = (a.Hq + a.Hkv) * 8;
#pragma unroll 4
      for (int32_t j = lane; j < nunit; j += 32) {
        const int32_t hh = j >> 3;
        const bool isq = hh < a.Hq;
        const size_t row = isq ? static_cast<size_t>(tok) * a.Hq + hh
                               : static_cast<size_t>(tok) * a.Hkv + (hh - a.Hq);
        uint4 v = *reinterpret_cast<const uint4 *>((isq ? a.q : a.k) + row * kDqk + 8 * cc);
        v.x = pack_bf16x2(bf16lo(v.x) * c0 - bf16hi(v.x) * s0, bf16lo(v.x) * s0 + bf16hi(v.x) * c0);
        v.y = pack_bf16x2(bf16lo(v.y) * c1 - bf16hi(v.y) * s1, bf16lo(v.y) * s1 + bf16hi(v.y) * c1);
        v.z = pack_bf16x2(bf16lo(v.z) * c2 - bf16hi(v.z) * s2, bf16lo(v.z) * s2 + bf16hi(v.z) * c2);
        v.w = pack_bf16x2(bf16lo(v.w) * c3 - bf16hi(v.w) * s3, bf16lo(v.w) * s3 + bf16hi(v.w) * c3);
        if (SA_IN(row, static_cast<int64_t>(a.total) * (isq ? a.Hq : a.Hkv), 0x30))
          *reinterpret_cast<uint4 *>((isq ? a.q_rot : a.k_rot) + row * 64 + 8 * cc) = v;
      }
    } else if (a.rope_on) {
      // pairs (t, t + 32): lane t holds pair t of every row
      float c, s;
      rope_cs(pos, a.rope_turns[lane], c, s);
#pragma unroll 4
      for (int32_t hh = 0; hh < a.Hq + a.Hkv; ++hh) {
        const bool isq = hh < a.Hq;
        const size_t row = isq ? static_cast<size_t>(tok) * a.Hq + hh
                               : static_cast<size_t>(tok) * a.Hkv + (hh - a.Hq);
        if (!SA_IN(row, static_cast<int64_t>(a.total) * (isq ? a.Hq : a.Hkv), 0x30)) continue;
        const __nv_bfloat16 *src = (isq ? a.q : a.k) + row * kDqk;
        __nv_bfloat16 *dst = (isq ? a.q_rot : a.k_rot) + row * 64;
        const float x = __bfloat162float(src[lane]), y = __bfloat162float(src[lane + 32]);
        dst[lane] = __float2bfloat16_rn(x * c - y * s);
        dst[lane + 32] = __float2bfloat16_rn(x * s + y * c);
      }
    }
    // D = dO . o per head: four lanes a head (32 dims each, 16-byte loads),
    // eight heads per round
    const int32_t quarter = lane & 3;
#pragma unroll 2
    for (int32_t h0 = 0; h0 < a.Hq; h0 += 8) {
      const int32_t h = h0 + (lane >> 2);
      float acc = 0.f;
      if (h < a.Hq) {
        const size_t row = static_cast<size_t>(tok) * a.Hq + h;
        const uint4 *op = reinterpret_cast<const uint4 *>(a.out + row * kDv + 32 * quarter);
        const uint4 *dp = reinterpret_cast<const uint4 *>(a.dout + row * kDv + 32 * quarter);
#pragma unroll
        for (int32_t u = 0; u < 4; ++u) {
          const uint4 ov = op[u], dv = dp[u];
          acc += bf16lo(ov.x) * bf16lo(dv.x) + bf16hi(ov.x) * bf16hi(dv.x);
          acc += bf16lo(ov.y) * bf16lo(dv.y) + bf16hi(ov.y) * bf16hi(dv.y);
          acc += bf16lo(ov.z) * bf16lo(dv.z) + bf16hi(ov.z) * bf16hi(dv.z);
          acc += bf16lo(ov.w) * bf16lo(dv.w) + bf16hi(ov.w) * bf16hi(dv.w);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (quarter == 0 && h < a.Hq &&
          SA_IN(static_cast<size_t>(tok) * a.Hq + h, static_cast<int64_t>(a.total) * a.Hq, 0x31)) {
        a.D[static_cast<size_t>(tok) * a.Hq + h] = acc;
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
    if (SA_IN(static_cast<size_t>(blockIdx.x) * a.Hq + h, static_cast<int64_t>(a.n_chunks) * a.Hq,
              0x32))
      a.dsink_part[static_cast<size_t>(blockIdx.x) * a.Hq + h] = acc;
  }
}

// One CTA per head: thread i sums the chunks i, i + 256, ... in order, then a
// fixed tree adds the 256 sums (the same bits every run).
__global__ void __launch_bounds__(256) bwd_dsink_kernel(const __grid_constant__ BwdArgs a) {
  __shared__ float part[256];
  const int32_t h = blockIdx.x;
  float acc = 0.f;
  for (int32_t c = threadIdx.x; c < a.n_chunks; c += 256)
    acc += a.dsink_part[static_cast<size_t>(c) * a.Hq + h];
  part[threadIdx.x] = acc;
  __syncthreads();
#pragma unroll
  for (int32_t w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0 && SA_OUT(h, a.Hq, 0x33)) a.dsink[h] = part[0];
}

// ------------------------------------------------------------------ shared pieces
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

// The same with the 32 angles of this row's position given, (cos, sin) of
// pair t at cs[t] (shared memory: the rows of one token share them).  One
// instance per pairing style, so the index pattern is fixed at compile time
// and x stays in registers.
template <int32_t kStyle>
__device__ __forceinline__ void bwd_unrotate_cs_t(float (&x)[64], const float2 *cs) {
  const float4 *cs4 = reinterpret_cast<const float4 *>(cs);
#pragma unroll
  for (int32_t t2 = 0; t2 < 16; ++t2) {
    const float4 a = cs4[t2];  // pairs 2 t2 and 2 t2 + 1
#pragma unroll
    for (int32_t e = 0; e < 2; ++e) {
      const int32_t t = 2 * t2 + e;
      const float c = e ? a.z : a.x, sn = e ? a.w : a.y;
      constexpr bool kInter = kStyle == 0;
      const int32_t i0 = kInter ? 2 * t : t, i1 = kInter ? 2 * t + 1 : t + 32;
      const float u = x[i0], w = x[i1];
      x[i0] = u * c + w * sn;
      x[i1] = w * c - u * sn;
    }
  }
}
__device__ __forceinline__ void bwd_unrotate_cs(float (&x)[64], int32_t style, const float2 *cs) {
  if (style == 0) bwd_unrotate_cs_t<0>(x, cs);
  else bwd_unrotate_cs_t<1>(x, cs);
}

// Gradient epilogues write 64-dim lines (128 bytes) of rows.  The four threads
// of a lane quad hold the same line of four rows, as 32 packed bf16 pairs each
// (w[8 s .. 8 s + 7] = sector s, 16 dims).  A 4 x 4 exchange of sectors inside
// the quad leaves in thread q sector q of rows 0..3 of the quad, so store j of
// the quad writes the whole line of row j: every store instruction moves whole
// 128-byte lines instead of a 16-byte piece of 32 lines.  All 32 lanes take
// part (the exchange is a warp shuffle); `line(j)` gives where row j's line
// starts, or null for a row that is not written.
template <class LineOf>
__device__ __forceinline__ void bwd_store_line_quad(uint32_t (&w)[32], LineOf line, bool v8) {
  const int32_t q = threadIdx.x & 3;
#pragma unroll
  for (int32_t j = 0; j < 2; ++j) {  // partner q ^ 2: sectors {0,1} <-> {2,3}
#pragma unroll
    for (int32_t e = 0; e < 8; ++e) {
      const uint32_t send = (q & 2) ? w[8 * j + e] : w[8 * (j + 2) + e];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
      if (q & 2) w[8 * j + e] = recv; else w[8 * (j + 2) + e] = recv;
    }
  }
#pragma unroll
  for (int32_t j = 0; j < 4; j += 2) {  // partner q ^ 1: positions j <-> j + 1
#pragma unroll
    for (int32_t e = 0; e < 8; ++e) {
      const uint32_t send = (q & 1) ? w[8 * j + e] : w[8 * (j + 1) + e];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
      if (q & 1) w[8 * j + e] = recv; else w[8 * (j + 1) + e] = recv;
    }
  }
#pragma unroll
  for (int32_t j = 0; j < 4; ++j) {
    __nv_bfloat16 *dst = line(j);
    if (dst == nullptr) continue;
    uint32_t (&sec)[8] = *reinterpret_cast<uint32_t(*)[8]>(w + 8 * j);
    if (v8) {
      st_global_v8(dst + 16 * q, sec);
    } else {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + 16 * q);
      d4[0] = make_uint4(sec[0], sec[1], sec[2], sec[3]);
      d4[1] = make_uint4(sec[4], sec[5], sec[6], sec[7]);
    }
  }
}

// Lines [l0, l0 + nl) of a gradient row held in TMEM from column t_col (fp32,
// this thread's lane): * scale, inverse RoPE on line 0 (dims 0..63, at
// position pos; angles from cs when given) when rope_on, bf16, stored through
// bwd_store_line_quad.
template <class LineOf>
__device__ __forceinline__ void bwd_store_lines(uint32_t t_col, int32_t l0, int32_t nl, float scale,
                                                bool rope_on, int32_t style, int32_t pos,
                                                const unsigned long long *turns, LineOf line,
                                                bool v8, const float2 *cs = nullptr) {
#pragma unroll 1
  for (int32_t l = l0; l < l0 + nl; ++l) {
    uint32_t r[64];
    tmem_ld32p(t_col + 64 * l, r);
    tmem_ld32p(t_col + 64 * l + 32, r + 32);
    tmem_wait_ld();
    reg_fence<64>(r);
    float x[64];
#pragma unroll
    for (int32_t e = 0; e < 64; ++e) x[e] = __uint_as_float(r[e]) * scale;
    if (l == 0 && rope_on) {
      if (cs != nullptr) bwd_unrotate_cs(x, style, cs);
      else bwd_unrotate(x, pos, style, turns);
    }
    uint32_t w[32];
#pragma unroll
    for (int32_t e = 0; e < 32; ++e) w[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
    bwd_store_line_quad(w, [&](int32_t j) { return line(j, l); }, v8);
  }
}

// ------------------------------------------------------------------ dQ kernel
// Work item of the dq kernel: one tile of 128/G query tokens x G heads of one
// KV head, over the 64-key blocks [lo, hi] its rows see.
struct DqItem {
  int32_t s0, L, t0, lo, nblk, kvh;
  bool valid;
};

__device__ __forceinline__ DqItem dq_item(const BwdArgs &a, int32_t it) {
  DqItem d{};
  d.valid = false;
  const int32_t T = 128 / a.G;
  const int32_t per_seq = a.Hkv * a.dq_tiles;
  const int32_t b = it / per_seq, rem = it % per_seq;
  d.kvh = rem % a.Hkv;
  // global: tiles in order (windowed) or longest first (causal)
  const int32_t tile = a.window > 0 ? rem / a.Hkv : a.dq_tiles - 1 - rem / a.Hkv;
  d.s0 = __ldg(a.cu_seqlens + b);
  d.L = __ldg(a.cu_seqlens + b + 1) - d.s0;
  d.t0 = tile * T;
  if (d.t0 >= d.L) return d;
  d.lo = a.window > 0 ? max(0, d.t0 - a.window + 1) : 0;
  const int32_t hi = min(d.L, d.t0 + T) - 1;
  d.nblk = (hi - d.lo + kDqBN) / kDqBN;
  d.valid = true;
  return d;
}

// The first item at or after `it` (stride gridDim.x) that has rows; `d` gets
// it (d.valid false when the CTA has no more).
__device__ __forceinline__ int32_t dq_next_item(const BwdArgs &a, int32_t it, DqItem &d) {
  d.valid = false;
  for (; it < a.dq_items; it += gridDim.x) {
    d = dq_item(a, it);
    if (d.valid) break;
  }
  return it;
}

struct DqLayout {
  static constexpr int32_t kStages = 3;                  // K/V blocks in flight
  static constexpr uint32_t kQBox = 128 * kRowBytes;     // 128 rows x 64 dims: 16 KB
  static constexpr uint32_t kKBox = kDqBN * kRowBytes;   // 64 keys x 64 dims: 8 KB
  static constexpr uint32_t kQOff = 0;                   // q_rot tile: 3 boxes
  static constexpr uint32_t kDoOff = 3 * kQBox;          // dO tile: 2 boxes
  static constexpr uint32_t kStOff = 5 * kQBox;          // stages: K 3 boxes, V 2 boxes
  static constexpr uint32_t kStage = 5 * kKBox;
  // qf, kv_full[3], kv_empty[3], mm1[2], q_empty, acc_full, ds_ready[2], drain
  static constexpr uint32_t kBarOff = kStOff + kStages * kStage;
  static constexpr uint32_t kMiscOff = kBarOff + 14 * 8;  // tmem slot, abort flag
  // RoPE angles of the epilogue: 4 warps x 4 tokens x 32 pairs of (cos, sin)
  static constexpr uint32_t kAngOff = kMiscOff + 16;
  static constexpr uint32_t kBytes = kAngOff + 4 * 4 * 32 * 8;
  static constexpr uint32_t kDynSmem = kBytes + 1024;
};
static_assert(DqLayout::kDynSmem <= 232448, "dq kernel shared memory");
// TMEM of the dq kernel: S and dP of key block g in buffer g & 1 (S at 128 b,
// dP at 128 b + 64), the dQ accumulator at 256..447.
constexpr uint32_t kDqColAcc = 256;

// Roles of the dq kernel, which meet only on mbarriers (block g is the g-th key
// block this CTA works on, over all its items):
//   copy thread (288): the Q/dO tile of an item and the K/V blocks, through
//     three stages; a stage is refilled once the dQ that read it is done
//     (KV_EMPTY); the next item's Q/dO once the last S/dP of the item is done
//     (Q_EMPTY).
//   MMA thread (256): S(g+1), dP(g+1) go out before dQ(g), so the tensor core
//     works while the rows turn S(g), dP(g) into dS(g); dQ(g) waits for all
//     256 row threads to have written dS(g) (DS_READY); after an item's last
//     dQ it hands the accumulator to the rows (ACC_FULL).
//   rows (0..255, two threads per packed query row, 32 keys each): dS into
//     TMEM over their own S columns, then at the end of an item the epilogue.
//     The first dQ of the next item needs these threads' DS_READY arrivals,
//     which come after their epilogue, so the accumulator is free by then.
// Q_EMPTY and ACC_FULL complete once per item: a wait on a barrier that
// completes per block could find it two phases behind (its parity would then
// match at once).
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q0,
                  const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ BwdArgs a) {
  using Ly = DqLayout;
  constexpr int32_t NS = Ly::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int32_t warp = threadIdx.x >> 5;
  const int32_t row = threadIdx.x & 127;  // packed query row == TMEM lane
  const int32_t half = threadIdx.x >> 7;    // this thread's 32 keys of a block
  const bool compute = threadIdx.x < 256;
  const bool issuer = threadIdx.x == 256;    // MMAs
  const bool producer = threadIdx.x == 288;  // copies
  auto bar = [&](uint32_t i) { return sbase + Ly::kBarOff + 8 * i; };
  const uint32_t B_QF = bar(0);
  auto B_KV = [&](uint32_t s) { return bar(1 + s); };
  auto B_KVE = [&](uint32_t s) { return bar(1 + NS + s); };
  auto B_MM1 = [&](uint32_t b) { return bar(1 + 2 * NS + b); };
  const uint32_t B_QE = bar(3 + 2 * NS), B_ACCF = bar(4 + 2 * NS);
  auto B_DSR = [&](uint32_t b) { return bar(5 + 2 * NS + b); };
  const uint32_t B_DRAIN = bar(7 + 2 * NS);
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  if (issuer) {
    mbar_init(B_QF, 1);
    for (uint32_t s = 0; s < static_cast<uint32_t>(NS); ++s) {
      mbar_init(B_KV(s), 1);
      mbar_init(B_KVE(s), 1);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(B_MM1(b), 1);
      mbar_init(B_DSR(b), 256);
    }
    mbar_init(B_QE, 1);
    mbar_init(B_ACCF, 1);
    mbar_init(B_DRAIN, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_q0);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_k0);
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
  const int32_t G = a.G;

  if (producer) {
    // ============================================================ copies
    DqItem ld;
    int32_t ld_it = dq_next_item(a, blockIdx.x, ld), ld_j = 0;
    uint32_t ld_g = 0, n_q = 0, n_done = 0;  // n_done: items whose blocks are all loaded
    auto load_q = [&](const DqItem &d) {
      mbar_arrive_expect_tx(B_QF, 5 * Ly::kQBox);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc)
        tma_load_3d(sbase + Ly::kQOff + cc * Ly::kQBox, cc ? &tm_q : &tm_q0, cc * 64, d.kvh * G,
                    d.s0 + d.t0, B_QF);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(sbase + Ly::kDoOff + cc * Ly::kQBox, &tm_do, cc * 64, d.kvh * G, d.s0 + d.t0, B_QF);
      ++n_q;
    };
    if (ld.valid) load_q(ld);
    while (ld.valid) {
      const uint32_t st = ld_g % NS;
      // the stage's previous block: its dQ is done
      if (ld_g >= static_cast<uint32_t>(NS) &&
          !wait_bar(B_KVE(st), ((ld_g / NS) & 1) ^ 1, abort_flag, 23))
        break;
      const uint32_t dst = sbase + Ly::kStOff + st * Ly::kStage;
      const int32_t krow = ld.s0 + ld.lo + ld_j * kDqBN;
      mbar_arrive_expect_tx(B_KV(st), Ly::kStage);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc)
        tma_load_3d(dst + cc * Ly::kKBox, cc ? &tm_k : &tm_k0, cc * 64, ld.kvh, krow, B_KV(st));
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(dst + (3 + cc) * Ly::kKBox, &tm_v, cc * 64, ld.kvh, krow, B_KV(st));
      ++ld_g;
      if (++ld_j >= ld.nblk) {
        ld_j = 0;
        ld_it = dq_next_item(a, ld_it + gridDim.x, ld);
        if (ld.valid) {
          // the item's last S/dP done: the Q/dO tile is free
          if (!wait_bar(B_QE, n_done & 1, abort_flag, 22)) break;
          load_q(ld);
        }
        ++n_done;
      }
    }
    // no copy may still be landing when shared memory goes back
    if (n_q > 0) drain_wait(B_QF, (n_q - 1) & 1);
    for (uint32_t s = 0; s < static_cast<uint32_t>(NS); ++s)
      if (ld_g > s) drain_wait(B_KV(s), ((ld_g - 1 - s) / NS) & 1);
  } else if (issuer) {
    // ============================================================ MMAs
    const uint32_t q_lo = ((sbase + Ly::kQOff) >> 4) | (1u << 16);
    const uint32_t do_lo = ((sbase + Ly::kDoOff) >> 4) | (1u << 16);
    constexpr uint32_t kIdS = idesc_f32acc(128, kDqBN, 1, 0, 0);
    constexpr uint32_t kIdQ = idesc_f32acc(128, kDqk, 1, 0, 1);
    // S(g) = Q K^T and dP(g) = dO V^T into buffer g & 1
    auto issue_sdp = [&](uint32_t g) -> bool {
      const uint32_t st = g % NS, buf = g & 1;
      if (!wait_bar(B_KV(st), (g / NS) & 1, abort_flag, 21)) return false;
      tc_fence_after();
      const uint32_t k_lo = ((sbase + Ly::kStOff + st * Ly::kStage) >> 4) | (1u << 16);
      const uint32_t v_lo = k_lo + ((3 * Ly::kKBox) >> 4);
#pragma unroll
      for (int ks = 0; ks < kDqk / 16; ++ks) {
        const uint32_t ao = ((ks >> 2) * Ly::kQBox + (ks & 3) * 32) >> 4;
        const uint32_t bo = ((ks >> 2) * Ly::kKBox + (ks & 3) * 32) >> 4;
        mma_ss2(tmem + buf * 128, q_lo + ao, kBwdDescHi, k_lo + bo, kBwdDescHi, kIdS, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < kDv / 16; ++ks) {
        const uint32_t ao = ((ks >> 2) * Ly::kQBox + (ks & 3) * 32) >> 4;
        const uint32_t bo = ((ks >> 2) * Ly::kKBox + (ks & 3) * 32) >> 4;
        mma_ss2(tmem + buf * 128 + 64, do_lo + ao, kBwdDescHi, v_lo + bo, kBwdDescHi, kIdS, ks > 0);
      }
      mma_commit(B_MM1(buf));
      return true;
    };
    DqItem cur;
    int32_t it = dq_next_item(a, blockIdx.x, cur);
    uint32_t g0 = 0, k = 0;
    bool ok = true, issued = false;
    while (ok && cur.valid) {
      if (!(ok = wait_bar(B_QF, k & 1, abort_flag, 20))) break;
      tc_fence_after();
      if (!(ok = issue_sdp(g0))) break;
      issued = true;
      if (cur.nblk == 1) mma_commit(B_QE);
      for (int32_t j = 0; j < cur.nblk; ++j) {
        const uint32_t g = g0 + j;
        if (j + 1 < cur.nblk) {
          if (!(ok = issue_sdp(g + 1))) break;
          if (j + 2 == cur.nblk) mma_commit(B_QE);  // the item's last S/dP
        }
        // all 256 row threads wrote dS(g)
        if (!(ok = wait_bar(B_DSR(g & 1), (g >> 1) & 1, abort_flag, 25))) break;
        tc_fence_after();
        const uint32_t st = g % NS;
        // A = dS: keys 16 ks.. of the block sit at columns 32 (ks / 2) + 8 (ks % 2)
#pragma unroll
        for (int ks = 0; ks < kDqBN / 16; ++ks)
          mma_ts2(tmem + kDqColAcc, tmem + (g & 1) * 128 + (ks >> 1) * 32 + (ks & 1) * 8,
                  ((sbase + Ly::kStOff + st * Ly::kStage) >> 4) + ks * ((16 * kRowBytes) >> 4) +
                      ((Ly::kKBox >> 4) << 16),
                  kBwdDescHi, kIdQ, (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(B_KVE(st));
        if (j + 1 == cur.nblk) mma_commit(B_ACCF);
      }
      g0 += cur.nblk;
      ++k;
      it = dq_next_item(a, it + gridDim.x, cur);
    }
    // every MMA done before TMEM goes back
    if (issued) {
      mma_commit(B_DRAIN);
      drain_wait(B_DRAIN, 0);
    }
  } else if (compute) {
    // ============================================================ rows
    const uint32_t lane_t = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int32_t t_row = row / G, g_row = row % G;
    // this row's lse and D in an item, loaded one item ahead (before the
    // epilogue) as they are, from a row that exists (row 0 for a row past the
    // end): nothing uses the loaded values before the next item starts, so
    // the loads never hold a thread up
    auto fetch_rows = [&](const DqItem &d, float &l_raw, float &d_raw) {
      const int32_t ti = d.t0 + t_row;
      const size_t grow =
          ti < d.L ? static_cast<size_t>(d.s0 + ti) * a.Hq + d.kvh * G + g_row : 0;
      l_raw = __ldg(a.lse + grow);
      d_raw = __ldg(a.D + grow);
    };
    DqItem cur;
    int32_t it = dq_next_item(a, blockIdx.x, cur);
    float l_raw = 0.f, d_raw = 0.f;
    if (cur.valid) fetch_rows(cur, l_raw, d_raw);
    uint32_t g0 = 0, k = 0;
    bool ok = true;
    while (ok && cur.valid) {
      const int32_t ti = cur.t0 + t_row;
      const bool rvalid = ti < cur.L;  // both halves of the row
      const float lse2 = rvalid ? l_raw * kLog2e : 0.f;
      const float Drow = rvalid ? d_raw : 0.f;
      for (int32_t j = 0; j < cur.nblk; ++j) {
        const uint32_t g = g0 + j;
        // S(g), dP(g) complete
        if (!(ok = wait_bar_warp(B_MM1(g & 1), (g >> 1) & 1, abort_flag, 22))) break;
        tc_fence_after();
        const uint32_t cs = lane_t + (g & 1) * 128 + 32 * half;
        uint32_t sv[32], pv[32];
        tmem_ld32p(cs, sv);
        tmem_ld32p(cs + 64, pv);
        tmem_wait_ld();
        reg_fence<32>(sv);
        reg_fence<32>(pv);
        // this row sees keys [max(0, ti - W + 1), ti]: columns c with
        // c - c_lo <= span (unsigned) of this half block
        const int32_t kb = cur.lo + j * kDqBN + 32 * half;
        const int32_t c_lo = (a.window > 0 ? ti - a.window + 1 : 0) - kb;
        const uint32_t span = rvalid ? static_cast<uint32_t>(ti - kb - c_lo) : 0u;
        // every row of the warp sees all 32 columns: no per-element mask
        const bool whole = __all_sync(0xffffffffu, rvalid && c_lo <= 0 && ti - kb >= 31);
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 nl2 = make_float2(-lse2, -lse2), nd2 = make_float2(-Drow, -Drow);
#pragma unroll
        for (int32_t c = 0; c < 32; c += 2) {
          const float2 y =
              ffma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, nl2);
          float2 p = make_float2(ex2(y.x), ex2(y.y));
          if (!whole) {
            if (!(static_cast<uint32_t>(c - c_lo) <= span && rvalid)) p.x = 0.f;
            if (!(static_cast<uint32_t>(c + 1 - c_lo) <= span && rvalid)) p.y = 0.f;
          }
          const float2 ds = fmul2(
              p, fadd2(make_float2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])), nd2));
          sv[c >> 1] = pack_bf16x2(ds.x, ds.y);
        }
        // dS of this half (16 bf16 pairs) over the first 16 of its own S columns
        tmem_st16p(cs, sv);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(B_DSR(g & 1));
      }
      if (!ok) break;
      DqItem nxt;
      const int32_t it_n = dq_next_item(a, it + gridDim.x, nxt);
      if (nxt.valid) fetch_rows(nxt, l_raw, d_raw);
      // the item's last dQ complete
      if (!(ok = wait_bar_warp(B_ACCF, k & 1, abort_flag, 24))) break;
      tc_fence_after();
      // dQ rows: line 0 (inverse RoPE) by the first thread of a row, lines 1
      // and 2 by the second
      const int32_t quad0 = row & ~3;
      auto line = [&](int32_t j, int32_t l) -> __nv_bfloat16 * {
        const int32_t r = quad0 + j, tj = cur.t0 + r / G;
        const size_t gr = static_cast<size_t>(cur.s0 + tj) * a.Hq + cur.kvh * G + r % G;
        if (tj >= cur.L || !SA_OUT(gr, static_cast<int64_t>(a.total) * a.Hq, 0x34)) return nullptr;
        return a.dq + gr * kDqk + 64 * l;
      };
      // line 0's inverse rotation: the G >= 8 rows of a token share its 32
      // angles, so its lanes compute 32 / min(G, 32) of them each and the warp
      // reads them back from shared memory
      const float2 *cs = nullptr;
      if (half == 0 && a.rope_on && G >= 8) {
        const int32_t lane = threadIdx.x & 31, Gw = min(G, 32);
        float2 *ang = reinterpret_cast<float2 *>(smem + Ly::kAngOff) + (warp * 4 + lane / Gw) * 32;
        __syncwarp();  // the previous item's angles are read
        for (int32_t p = lane % Gw; p < 32; p += Gw) {
          float c, sn;
          rope_cs(ti, a.rope_turns[p], c, sn);
          ang[p] = make_float2(c, sn);
        }
        __syncwarp();
        cs = ang;
      }
      bwd_store_lines(lane_t + kDqColAcc, half == 0 ? 0 : 1, half == 0 ? 1 : 2, a.scale, a.rope_on,
                      a.rope_style, ti, a.rope_turns, line, a.grad_v8 != 0, cs);
      tc_fence_before();
      g0 += cur.nblk;
      ++k;
      cur = nxt;
      it = it_n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dK / dV kernel
// Work item of the dk/dv kernel: one block of 128 keys of one KV head, over the
// sub-tiles of 64 packed query rows (64/G tokens x G heads) that see it.
struct KvItem {
  int32_t s0, L, k0, i_lo, nsub, kvh;
  bool valid;
};

__device__ __forceinline__ KvItem kv_item(const BwdArgs &a, int32_t it) {
  KvItem d{};
  d.valid = false;
  const int32_t TS = kKvRows / a.G;
  const int32_t per_seq = a.Hkv * a.kv_blocks;
  const int32_t b = it / per_seq, rem = it % per_seq;
  d.kvh = rem % a.Hkv;
  const int32_t blk = rem / a.Hkv;  // global: the earliest blocks (most queries) first
  d.s0 = __ldg(a.cu_seqlens + b);
  d.L = __ldg(a.cu_seqlens + b + 1) - d.s0;
  d.k0 = blk * kKvBN;
  if (d.k0 >= d.L) return d;
  d.i_lo = d.k0;
  const int32_t i_hi = a.window > 0 ? min(d.L - 1, d.k0 + kKvBN - 1 + a.window - 1) : d.L - 1;
  d.nsub = (i_hi - d.i_lo + TS) / TS;
  d.valid = true;
  return d;
}

__device__ __forceinline__ int32_t kv_next_item(const BwdArgs &a, int32_t it, KvItem &d) {
  d.valid = false;
  for (; it < a.kv_items; it += gridDim.x) {
    d = kv_item(a, it);
    if (d.valid) break;
  }
  return it;
}

struct KvLayout {
  static constexpr int32_t kStages = 3;                  // Q/dO sub-tiles in flight
  static constexpr uint32_t kKBox = kKvBN * kRowBytes;   // 128 keys x 64 dims: 16 KB
  static constexpr uint32_t kQBox = kKvRows * kRowBytes; // 64 rows x 64 dims: 8 KB
  static constexpr uint32_t kKOff = 0;                   // k_rot block: 3 boxes
  static constexpr uint32_t kVOff = 3 * kKBox;           // v block: 2 boxes
  static constexpr uint32_t kStOff = 5 * kKBox;          // stages: q_rot rows 3 boxes, dO rows 2
  static constexpr uint32_t kStage = 5 * kQBox;
  static constexpr uint32_t kColOff = kStOff + kStages * kStage;  // lse*log2e, D: 2 sub-tiles
  // kv_full, kv_empty, qs_full[3], qs_empty[3], mm1, mm2, p_ready, acc_full, rows_full[2],
  // drain, s_read
  static constexpr uint32_t kBarOff = kColOff + 2 * 2 * kKvRows * 4;
  static constexpr uint32_t kMiscOff = kBarOff + 16 * 8;
  static constexpr uint32_t kBytes = kMiscOff + 16;
  static constexpr uint32_t kDynSmem = kBytes + 1024;
};
static_assert(KvLayout::kDynSmem <= 232448, "dkdv kernel shared memory");

// Roles of the dk/dv kernel, which meet only on mbarriers (sub-tile g is the
// g-th query sub-tile this CTA works on, over all its items).  TMEM: S^T 0..63
// and dP^T 64..127 of the current sub-tile, dV 128..255, dK 256..447, and P^T
// (448..479) and dS^T (480..511) as bf16 pairs.
//   copy thread (288): the K/V block of an item once the previous item's last
//     S^T/dP^T is done (KV_EMPTY); Q/dO sub-tiles, last query rows first (so
//     the CTAs of one KV head stream the same rows together), through three
//     stages, each refilled once the dV/dK that read it is done (QS_EMPTY).
//   MMA thread (256): once every row has S^T/dP^T(g) in registers (S_READ),
//     S^T/dP^T(g+1) go out, so the tensor core computes them while the rows
//     turn sub-tile g into P^T/dS^T; once those are in TMEM (P_READY),
//     dV/dK(g) follow; after an item's last dV/dK it hands the accumulators
//     over (ACC_FULL).  The first S^T/dP^T of an item goes out after the
//     previous item's last P_READY, which also means its S^T/dP^T were read.
//   rows (0..255, two threads per key, 32 query rows each): they wait for
//     dV/dK(g-1) only before writing P^T/dS^T(g).  Rows 0..63 load lse and D of
//     the next sub-tile at the top of a sub-tile and put them in a
//     shared-memory slot after that wait (ROWS_FULL): by then every row has
//     read the slot's previous contents (dV/dK(g-1) needed all their
//     P_READY arrivals for sub-tile g-1).
// KV_EMPTY and ACC_FULL complete once per item, so no wait can find its
// barrier two phases away from the awaited one.
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q0,
                    const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ BwdArgs a) {
  using Ly = KvLayout;
  constexpr int32_t NS = Ly::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int32_t warp = threadIdx.x >> 5;
  const int32_t lane_row = threadIdx.x & 127;  // key row == TMEM lane
  const int32_t half = threadIdx.x >> 7;         // this thread's 32 query rows of a sub-tile
  const bool compute = threadIdx.x < 256;
  const bool issuer = threadIdx.x == 256;    // MMAs
  const bool producer = threadIdx.x == 288;  // copies
  auto bar = [&](uint32_t i) { return sbase + Ly::kBarOff + 8 * i; };
  const uint32_t B_KF = bar(0), B_KVE = bar(1);
  auto B_QS = [&](uint32_t s) { return bar(2 + s); };
  auto B_QSE = [&](uint32_t s) { return bar(2 + NS + s); };
  const uint32_t B_MM1 = bar(2 + 2 * NS), B_MM2 = bar(3 + 2 * NS);
  const uint32_t B_PR = bar(4 + 2 * NS), B_ACCF = bar(5 + 2 * NS);
  auto B_LF = [&](uint32_t p) { return bar(6 + 2 * NS + p); };
  const uint32_t B_DRAIN = bar(8 + 2 * NS), B_SR = bar(9 + 2 * NS);
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  float *c_lse = reinterpret_cast<float *>(smem + Ly::kColOff);  // [2][64]
  float *c_D = c_lse + 2 * kKvRows;                                // [2][64]
  if (issuer) {
    mbar_init(B_KF, 1);
    mbar_init(B_KVE, 1);
    for (uint32_t s = 0; s < static_cast<uint32_t>(NS); ++s) {
      mbar_init(B_QS(s), 1);
      mbar_init(B_QSE(s), 1);
    }
    mbar_init(B_MM1, 1);
    mbar_init(B_MM2, 1);
    mbar_init(B_PR, 256);
    mbar_init(B_ACCF, 1);
    mbar_init(B_LF(0), kKvRows);
    mbar_init(B_LF(1), kKvRows);
    mbar_init(B_DRAIN, 1);
    mbar_init(B_SR, 256);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_q0);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_k0);
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
  const int32_t G = a.G, TS = kKvRows / G;  // tokens per sub-tile
  constexpr uint32_t kColST = 0, kColPT = 64, kColV = 128, kColK = 256, kColP = 448, kColDS = 480;
  // Sub-tile s of an item starts at query token sub0(d, s).  A query row is
  // seen by two neighbouring key blocks, whose items start together on
  // neighbouring CTAs; even blocks walk their sub-tiles from the last rows
  // down and odd blocks from the first rows up, so the two CTAs reading a
  // shared row read it a few sub-tiles apart and the second read hits L2
  // (walking both one way, they read it half an item apart: 2.77 against
  // 1.80 GB of DRAM reads on a 32768-token SWA layer).
  auto sub0 = [&](const KvItem &d, int32_t sidx) {
    return ((d.k0 / kKvBN) & 1) ? d.i_lo + sidx * TS : d.i_lo + (d.nsub - 1 - sidx) * TS;
  };

  if (producer) {
    // ============================================================ copies
    KvItem ld;
    int32_t ld_it = kv_next_item(a, blockIdx.x, ld), ld_j = 0;
    uint32_t ld_g = 0, n_kv = 0;
    auto load_kv = [&](const KvItem &d) {
      mbar_arrive_expect_tx(B_KF, 5 * Ly::kKBox);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc)
        tma_load_3d(sbase + Ly::kKOff + cc * Ly::kKBox, cc ? &tm_k : &tm_k0, cc * 64, d.kvh,
                    d.s0 + d.k0, B_KF);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(sbase + Ly::kVOff + cc * Ly::kKBox, &tm_v, cc * 64, d.kvh, d.s0 + d.k0, B_KF);
      ++n_kv;
    };
    while (ld.valid) {
      if (ld_j == 0) {
        // the previous item's last S^T/dP^T done: the K/V block is free
        if (n_kv > 0 && !wait_bar(B_KVE, (n_kv - 1) & 1, abort_flag, 24)) break;
        load_kv(ld);
      }
      const uint32_t st = ld_g % NS;
      // the stage's previous sub-tile: its dV/dK is done
      if (ld_g >= static_cast<uint32_t>(NS) &&
          !wait_bar(B_QSE(st), ((ld_g / NS) & 1) ^ 1, abort_flag, 23))
        break;
      const uint32_t dst = sbase + Ly::kStOff + st * Ly::kStage;
      const int32_t tok = ld.s0 + sub0(ld, ld_j);
      mbar_arrive_expect_tx(B_QS(st), Ly::kStage);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc)
        tma_load_3d(dst + cc * Ly::kQBox, cc ? &tm_q : &tm_q0, cc * 64, ld.kvh * G, tok, B_QS(st));
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(dst + (3 + cc) * Ly::kQBox, &tm_do, cc * 64, ld.kvh * G, tok, B_QS(st));
      ++ld_g;
      if (++ld_j >= ld.nsub) {
        ld_j = 0;
        ld_it = kv_next_item(a, ld_it + gridDim.x, ld);
      }
    }
    // no copy may still be landing when shared memory goes back
    if (n_kv > 0) drain_wait(B_KF, (n_kv - 1) & 1);
    for (uint32_t s = 0; s < static_cast<uint32_t>(NS); ++s)
      if (ld_g > s) drain_wait(B_QS(s), ((ld_g - 1 - s) / NS) & 1);
  } else if (issuer) {
    // ============================================================ MMAs
    const uint32_t k_lo = ((sbase + Ly::kKOff) >> 4) | (1u << 16);
    const uint32_t v_lo = ((sbase + Ly::kVOff) >> 4) | (1u << 16);
    constexpr uint32_t kIdS = idesc_f32acc(128, kKvRows, 1, 0, 0);
    constexpr uint32_t kIdV = idesc_f32acc(128, kDv, 1, 0, 1);
    constexpr uint32_t kIdK = idesc_f32acc(128, kDqk, 1, 0, 1);
    // S^T(g) = K Q^T and dP^T(g) = V dO^T
    auto issue_sdp = [&](uint32_t g) -> bool {
      const uint32_t st = g % NS;
      if (!wait_bar(B_QS(st), (g / NS) & 1, abort_flag, 25)) return false;
      tc_fence_after();
      const uint32_t q_lo = ((sbase + Ly::kStOff + st * Ly::kStage) >> 4) | (1u << 16);
      const uint32_t do_lo = q_lo + ((3 * Ly::kQBox) >> 4);
#pragma unroll
      for (int ks = 0; ks < kDqk / 16; ++ks) {
        const uint32_t ao = ((ks >> 2) * Ly::kKBox + (ks & 3) * 32) >> 4;
        const uint32_t bo = ((ks >> 2) * Ly::kQBox + (ks & 3) * 32) >> 4;
        mma_ss2(tmem + kColST, k_lo + ao, kBwdDescHi, q_lo + bo, kBwdDescHi, kIdS, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < kDv / 16; ++ks) {
        const uint32_t ao = ((ks >> 2) * Ly::kKBox + (ks & 3) * 32) >> 4;
        const uint32_t bo = ((ks >> 2) * Ly::kQBox + (ks & 3) * 32) >> 4;
        mma_ss2(tmem + kColPT, v_lo + ao, kBwdDescHi, do_lo + bo, kBwdDescHi, kIdS, ks > 0);
      }
      mma_commit(B_MM1);
      return true;
    };
    KvItem cur;
    int32_t it = kv_next_item(a, blockIdx.x, cur);
    uint32_t g0 = 0, k = 0;
    bool ok = true, issued = false;
    while (ok && cur.valid) {
      if (!(ok = wait_bar(B_KF, k & 1, abort_flag, 24))) break;
      tc_fence_after();
      if (!(ok = issue_sdp(g0))) break;
      issued = true;
      if (cur.nsub == 1) mma_commit(B_KVE);
      for (int32_t sidx = 0; sidx < cur.nsub; ++sidx) {
        const uint32_t g = g0 + sidx;
        // S^T/dP^T of the next sub-tile as soon as every row has S^T/dP^T(g)
        // in registers, so they run while the rows compute P^T/dS^T(g)
        if (sidx + 1 < cur.nsub) {
          if (!(ok = wait_bar(B_SR, g & 1, abort_flag, 29))) break;
          tc_fence_after();
          if (!(ok = issue_sdp(g + 1))) break;
          if (sidx + 2 == cur.nsub) mma_commit(B_KVE);  // the item's last S^T/dP^T
        }
        // the rows wrote P^T/dS^T(g): dV/dK(g)
        if (!(ok = wait_bar(B_PR, g & 1, abort_flag, 26))) break;
        tc_fence_after();
        const uint32_t stb = (sbase + Ly::kStOff + (g % NS) * Ly::kStage) >> 4;
#pragma unroll
        for (int ks = 0; ks < kKvRows / 16; ++ks) {
          const uint32_t step = ks * ((16 * kRowBytes) >> 4);
          // dV += P^T dO: B = the dO rows read N-major (LBO = one box)
          mma_ts2(tmem + kColV, tmem + kColP + ks * 8,
                  stb + ((3 * Ly::kQBox) >> 4) + step + ((Ly::kQBox >> 4) << 16), kBwdDescHi, kIdV,
                  (sidx > 0 || ks > 0) ? 1u : 0u);
          // dK += dS^T Q: B = the q_rot rows read N-major
          mma_ts2(tmem + kColK, tmem + kColDS + ks * 8, stb + step + ((Ly::kQBox >> 4) << 16),
                  kBwdDescHi, kIdK, (sidx > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(B_MM2);
        mma_commit(B_QSE(g % NS));
        if (sidx + 1 == cur.nsub) mma_commit(B_ACCF);
      }
      g0 += cur.nsub;
      ++k;
      it = kv_next_item(a, it + gridDim.x, cur);
    }
    // every MMA done before TMEM goes back
    if (issued) {
      mma_commit(B_DRAIN);
      drain_wait(B_DRAIN, 0);
    }
  } else if (compute) {
    // ============================================================ rows
    const uint32_t lane_t = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool writer = threadIdx.x < kKvRows;  // stages lse and D of one query row
    // the values as loaded (from row 0 for a row past the end) and whether
    // the row exists: nothing uses a loaded value until it is staged, after
    // the sub-tile's work, so the loads never hold the writer up
    float r_lse = 0.f, r_D = 0.f;
    bool r_v = false;
    auto fetch_rows = [&](const KvItem &d, int32_t sidx) {
      const int32_t ti = sub0(d, sidx) + threadIdx.x / G, h = d.kvh * G + threadIdx.x % G;
      r_v = ti < d.L;
      const size_t grow = r_v ? static_cast<size_t>(d.s0 + ti) * a.Hq + h : 0;
      r_lse = __ldg(a.lse + grow);
      r_D = __ldg(a.D + grow);
    };
    KvItem cur;
    int32_t it = kv_next_item(a, blockIdx.x, cur);
    if (cur.valid && writer) {
      fetch_rows(cur, 0);
      c_lse[threadIdx.x] = r_v ? r_lse * kLog2e : 0.f;
      c_D[threadIdx.x] = r_v ? r_D : 0.f;
      mbar_arrive(B_LF(0));
    }
    uint32_t g0 = 0, k = 0;
    bool ok = true;
    while (ok && cur.valid) {
      KvItem nxt;
      const int32_t it_n = kv_next_item(a, it + gridDim.x, nxt);
      const int32_t kj = cur.k0 + lane_row;  // this thread's key (both halves)
      const bool kvalid = kj < cur.L;
      for (int32_t sidx = 0; sidx < cur.nsub; ++sidx) {
        const uint32_t g = g0 + sidx;
        const int32_t i0 = sub0(cur, sidx);
        const bool more = sidx + 1 < cur.nsub || nxt.valid;
        // the next sub-tile's rows: the loads go out now
        if (writer && more) {
          if (sidx + 1 < cur.nsub)
            fetch_rows(cur, sidx + 1);
          else
            fetch_rows(nxt, 0);
        }
        // S^T(g), dP^T(g) complete; this sub-tile's lse and D in their slot
        if (!(ok = wait_bar_warp(B_MM1, g & 1, abort_flag, 22))) break;
        if (!(ok = wait_bar_warp(B_LF(g & 1), (g >> 1) & 1, abort_flag, 21))) break;
        tc_fence_after();
        const float4 *cl4 = reinterpret_cast<const float4 *>(c_lse + (g & 1) * kKvRows + 32 * half);
        const float4 *cd4 = reinterpret_cast<const float4 *>(c_D + (g & 1) * kKvRows + 32 * half);
        // column c is query token i0 + c / G: this key is seen by the columns
        // with i0 + c / G in [kj, min(L, kj + W) - 1], i.e. c in [c_lo, c_hi)
        // (token counts clamped to one sub-tile first, so no product overflows);
        // this thread takes columns 32 half .. 32 half + 31
        const int32_t d0 = kj - i0;
        const int32_t c_lo = (d0 > 0 ? d0 * G : 0) - 32 * half;
        int32_t c_hi = min(cur.L - i0, kKvRows) * G;
        if (a.window > 0) c_hi = min(c_hi, max(0, min(d0 + a.window, kKvRows)) * G);
        c_hi = min(c_hi, kKvRows) - 32 * half;
        const uint32_t span = (kvalid && c_hi > c_lo) ? static_cast<uint32_t>(c_hi - c_lo) : 0u;
        uint32_t sv[32], pv[32];
        tmem_ld32p(lane_t + kColST + 32 * half, sv);
        tmem_ld32p(lane_t + kColPT + 32 * half, pv);
        tmem_wait_ld();
        reg_fence<32>(sv);
        reg_fence<32>(pv);
        // S^T/dP^T(g) are in registers: their columns may take the next sub-tile's
        tc_fence_before();
        mbar_arrive(B_SR);
        // every key of the warp sees all 32 columns: no per-element mask
        const bool whole = __all_sync(
            0xffffffffu, kvalid && c_lo <= 0 && static_cast<int64_t>(span) > 31 - c_lo);
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
        for (int32_t c = 0; c < 32; c += 4) {
          const float4 l4 = cl4[c >> 2], d4 = cd4[c >> 2];
          const float2 nl[2] = {make_float2(-l4.x, -l4.y), make_float2(-l4.z, -l4.w)};
          const float2 nd[2] = {make_float2(-d4.x, -d4.y), make_float2(-d4.z, -d4.w)};
#pragma unroll
          for (int32_t h2 = 0; h2 < 2; ++h2) {
            const int32_t cc = c + 2 * h2;  // columns cc, cc + 1 (already read: 0 .. cc - 1)
            const float2 y =
                ffma2(make_float2(__uint_as_float(sv[cc]), __uint_as_float(sv[cc + 1])), sc2, nl[h2]);
            float2 p = make_float2(ex2(y.x), ex2(y.y));
            if (!whole) {
              if (!(static_cast<uint32_t>(cc - c_lo) < span)) p.x = 0.f;
              if (!(static_cast<uint32_t>(cc + 1 - c_lo) < span)) p.y = 0.f;
            }
            const float2 ds = fmul2(
                p, fadd2(make_float2(__uint_as_float(pv[cc]), __uint_as_float(pv[cc + 1])), nd[h2]));
            sv[cc >> 1] = pack_bf16x2(p.x, p.y);
            pv[cc >> 1] = pack_bf16x2(ds.x, ds.y);
          }
        }
        // dV/dK(g-1) complete: they have read P^T/dS^T(g-1), and every row
        // has read this CTA's other lse / D slot
        if (g > 0 && !(ok = wait_bar_warp(B_MM2, (g - 1) & 1, abort_flag, 27))) break;
        tc_fence_after();
        tmem_st16p(lane_t + kColP + 16 * half, sv);   // P^T as bf16 pairs
        tmem_st16p(lane_t + kColDS + 16 * half, pv);  // dS^T as bf16 pairs
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(B_PR);
        if (writer && more) {
          c_lse[((g + 1) & 1) * kKvRows + threadIdx.x] = r_v ? r_lse * kLog2e : 0.f;
          c_D[((g + 1) & 1) * kKvRows + threadIdx.x] = r_v ? r_D : 0.f;
          mbar_arrive(B_LF((g + 1) & 1));
        }
      }
      if (!ok) break;
      // the item's last dV/dK complete
      if (!(ok = wait_bar_warp(B_ACCF, k & 1, abort_flag, 28))) break;
      tc_fence_after();
      // dV rows (lines 0, 1) and line 2 of the dK rows by the first thread of
      // a key, dK lines 0 (inverse RoPE) and 1 by the second
      const int32_t quad0 = lane_row & ~3;
      auto kv_row = [&](int32_t j, int64_t &r) {
        const int32_t kk = cur.k0 + quad0 + j;
        r = static_cast<int64_t>(cur.s0 + kk) * a.Hkv + cur.kvh;
        return kk < cur.L;
      };
      auto dv_line = [&](int32_t j, int32_t l) -> __nv_bfloat16 * {
        int64_t r;
        if (!kv_row(j, r) || !SA_OUT(r, static_cast<int64_t>(a.total) * a.Hkv, 0x35)) return nullptr;
        return a.dv + r * kDv + 64 * l;
      };
      auto dk_line = [&](int32_t j, int32_t l) -> __nv_bfloat16 * {
        int64_t r;
        if (!kv_row(j, r) || !SA_OUT(r, static_cast<int64_t>(a.total) * a.Hkv, 0x36)) return nullptr;
        return a.dk + r * kDqk + 64 * l;
      };
      if (half == 0) {
        bwd_store_lines(lane_t + kColV, 0, 2, 1.f, false, 0, 0, a.rope_turns, dv_line,
                        a.grad_v8 != 0);
        bwd_store_lines(lane_t + kColK, 2, 1, a.scale, false, 0, 0, a.rope_turns, dk_line,
                        a.grad_v8 != 0);
      } else {
        bwd_store_lines(lane_t + kColK, 0, 2, a.scale, a.rope_on, a.rope_style, kj, a.rope_turns,
                        dk_line, a.grad_v8 != 0);
      }
      tc_fence_before();
      g0 += cur.nsub;
      ++k;
      cur = nxt;
      it = it_n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace sa
