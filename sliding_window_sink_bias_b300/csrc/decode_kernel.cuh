// decode_kernel.cuh -- split-KV partials of the multi-token (MTP-verify) decode.
//
// The MiMo-V2-Flash Technical Report (§2.3.1) verifies 1 + K draft tokens in
// one pass over the KV cache.  For each unit (sequence b, KV head) the T new
// tokens x G query heads of that KV head form T * G <= 128 packed rows, and the
// unit's visible keys are cut into 64-key blocks.  Each KV head has its own
// list of its units' blocks (sequence by sequence), cut into equal contiguous
// ranges over the same number of CTAs: every CTA streams the same number of
// cache blocks whatever the sequence lengths, and the CTAs of the different
// KV heads walk each sequence's cache rows together (a head's 384-byte key
// slice shares 256-byte DRAM bursts with its neighbours', so walking them at
// different times fetches those bursts twice).  A unit that lies entirely inside one CTA's range is finished there
// (eqs. (1)-(3) of §2.2, the sink added once); a unit cut by a range boundary
// leaves, per CTA, its running max m, the sum l of 2^(a - m) and the
// unnormalised O = sum 2^(a - m) v without the sink; the CTA whose arrival
// completes the unit's ticket (the last of its CTAs to finish it) merges the
// partials in a fixed order and adds the sink once, in the same launch.
//
// The cache is streamed in 64-key blocks, four in flight (TMA into a shared
// memory ring); S = Q K^T and O += P V run on tcgen05 with S, P and O in TMEM.
// Only the T * G packed rows that exist are touched by the softmax.
//
// Warp roles (384 threads, one CTA per SM):
//   warp 0       TMA producer: Q tile once per chunk, K/V blocks.
//   warp 1       MMA issuer: S = Q K^T (12 k-steps, Q from TMEM), then O += P V.
//   warp 2       TMEM allocator (S0, S1, O, Q: 512 columns).
//   warp 3       set-up: this CTA's block range and first unit; the rows of
//                its share of the units with no key at all.
//   warps 4-7    online softmax, one row per thread: the block's masked max
//                (3-input max), lazy running max (moves only when a block
//                exceeds it by more than 2^8), P = 2^(s * scale * log2e - m) as
//                bf16 pairs into TMEM, l, and the rescale of this row's O when
//                m moves; at the end of a unit's segment the row is finished
//                (with the sink) or its partial is written.
//   warps 8-11   RoPE on dims 0..63 of the Q tile, the tile into one of two
//                TMEM buffers (one row per thread), RoPE on every K block.
#pragma once
#include "common.cuh"

namespace sa {

constexpr int32_t kDecBN = 64;      // keys per block
constexpr int32_t kDecStages = 4;   // K/V blocks in flight
constexpr uint32_t kDecTmemCols = 512;
constexpr uint32_t kDecTmemO = 128;
// The units' query tiles (128 rows x 192 dims, 16-bit pairs: 96 columns), two
// buffers: QK^T reads its A operand from TMEM, so a tile is not re-read from
// shared memory for every cache block (with N = 64 keys, 48 KB of Q against
// 24 KB of K per block), and the next unit's tile goes in while QK^T still
// reads the current one.
__host__ __device__ constexpr uint32_t dec_tmem_q(uint32_t b) { return 256u + 96u * b; }
constexpr int32_t kDecMaxGrid = 160;  // CTAs at most (2 partial slots each)

struct DecArgs {
  int32_t Hq, Hkv, G, T;
  int32_t R;              // T * G packed rows
  int32_t window;
  int32_t batch, S_cap;
  int32_t n_units;        // batch * Hkv
  // The work is n_sub independent block lists of n_k units each (n_sub = Hkv:
  // one list per KV head, so the KV heads of a sequence stream its cache rows
  // at the same time; n_sub = 1: one list over all units).  Unit k of list s
  // is u = k * n_sub + s; CTA c works on list c % n_sub.
  int32_t n_sub, n_k;
  int32_t kv_ring;        // 1: the cache is a ring of S_cap slots, position j at slot j % S_cap
  int32_t k_rotated;      // 1: the cached keys are already rotated at their positions
  int32_t rope_on, rope_style;
  const float *k_scale, *v_scale;  // FP8 cache: per-KV-head dequantisation scales
  uint32_t q_tx_bytes;
  float scale_log2;       // > 0
  const int32_t *seqlens;
  const float *sink;
  __nv_bfloat16 *out;
  float *lse;
  // per-unit tickets of the units CTA ranges cut: (epoch << 16) | arrivals;
  // epoch is this call's number (48 bits), so a word another call left behind
  // just starts over and the workspace needs no clearing
  unsigned long long *tickets;
  unsigned long long epoch;
  float *part_o;          // [gridDim.x * 2, R, 128] unnormalised O
  float *part_ml;         // [gridDim.x * 2, R, 4] (m, l, 0, 0), log2 domain
  int64_t n_rows;         // rows of out and lse: B x T x Hq (checked stores)
  int64_t n_part_rows;    // rows the partial buffers hold (checked accesses)
  unsigned long long rope_turns[32];
};

// Visible keys of unit u = b * Hkv + kvh: [lo, L) with L = seqlens[b]; with a
// window only the last T + W - 1 keys can be seen by the T queries.
__device__ __forceinline__ void dec_unit_keys(const DecArgs &a, int32_t u, int32_t &L, int32_t &lo,
                                              int32_t &nblk) {
  L = __ldg(a.seqlens + u / a.Hkv);
  lo = a.window > 0 ? max(0, L - a.T - a.window + 1) : 0;
  // a ring cache is read in 16-key pieces that must not straddle the ring's
  // end: blocks start on a multiple of 16 (the keys before lo are masked)
  if (a.kv_ring) lo &= ~15;
  nblk = L > lo ? (L - lo + kDecBN - 1) / kDecBN : 0;
}

// One segment: blocks [blk0, blk0 + nblk) of unit u, processed by this CTA.
struct DecSeg {
  int32_t u, b, kvh, L, lo;
  int32_t blk0, nblk, nblk_u;
  int32_t first;  // the CTA's first segment (partial slot 0, else slot 1)
};

struct DecCursor {
  int32_t k, blk;  // next block to process: unit k of this CTA's list, block blk
  int32_t s;       // the list (unit u = k * n_sub + s)
  int32_t left;    // blocks of this CTA not yet handed out
  int32_t first;
};

// The next segment of the cursor (returns false when the CTA's range is done).
__device__ __forceinline__ bool dec_next(DecCursor &c, const DecArgs &a, DecSeg &sg) {
  while (c.left > 0 && c.k < a.n_k) {
    const int32_t u = c.k * a.n_sub + c.s;
    int32_t L, lo, nb;
    dec_unit_keys(a, u, L, lo, nb);
    if (c.blk >= nb) {
      ++c.k;
      c.blk = 0;
      continue;
    }
    sg.u = u;
    sg.b = u / a.Hkv;
    sg.kvh = u % a.Hkv;
    sg.L = L;
    sg.lo = lo;
    sg.nblk_u = nb;
    sg.blk0 = c.blk;
    sg.nblk = min(nb - c.blk, c.left);
    sg.first = c.first;
    c.first = 0;
    c.left -= sg.nblk;
    c.blk += sg.nblk;
    return true;
  }
  return false;
}

// Rows of unit u with no key at all (an empty cache): o = 0, lse = sink (the
// empty sum of eqs. (2)-(3)).  One warp.
__device__ void dec_write_empty_unit(const DecArgs &a, int32_t u, int32_t lane) {
  const int32_t b = u / a.Hkv, kvh = u % a.Hkv;
  for (int32_t r = 0; r < a.R; ++r) {
    const int32_t head = kvh * a.G + r % a.G;
    const size_t orow = (static_cast<size_t>(b) * a.T + r / a.G) * a.Hq + head;
    if (!SA_OUT(orow, a.n_rows, 0x20)) continue;
    reinterpret_cast<uint2 *>(a.out + orow * kDv)[lane] = make_uint2(0u, 0u);
    if (lane == 0) a.lse[orow] = __ldg(a.sink + head);
  }
}

// Set-up (one warp): the block counts of the units of this CTA's list (a warp
// scan), this CTA's range [f0, f1) of the list's blocks (the list's G =
// gridDim.x / n_sub CTAs split it evenly) and the unit/block it starts at.
// Units without keys are written here, unit k of the list by the list's CTA
// k % G.  cur: first unit, its first block, blocks of the range, list, the
// list's total blocks, f0.
__device__ void dec_locate(const DecArgs &a, int32_t lane, int32_t *cur) {
  const int32_t sl = static_cast<int32_t>(blockIdx.x) % a.n_sub;
  const int32_t g = static_cast<int32_t>(blockIdx.x) / a.n_sub;
  const int32_t G = static_cast<int32_t>(gridDim.x) / a.n_sub;
  int64_t run = 0;
  // pass 1: total blocks of the list; this CTA's share of the empty units
  for (int32_t base = 0; base < a.n_k; base += 32) {
    const int32_t k = base + lane;
    int32_t nb = 0;
    if (k < a.n_k) {
      int32_t L, lo;
      dec_unit_keys(a, k * a.n_sub + sl, L, lo, nb);
    }
    uint32_t empty = __ballot_sync(0xffffffffu, k < a.n_k && nb == 0 && k % G == g);
    while (empty) {
      const int32_t j = __ffs(empty) - 1;
      empty &= empty - 1;
      dec_write_empty_unit(a, (base + j) * a.n_sub + sl, lane);
    }
    int32_t incl = nb;
#pragma unroll
    for (int32_t o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  const int64_t T = run;
  const int64_t f0 = T * g / G;
  const int64_t f1 = T * (g + 1) / G;
  // pass 2: the unit holding block f0
  int32_t sk = a.n_k, sblk = 0;
  run = 0;
  bool found = false;
  for (int32_t base = 0; base < a.n_k && !found && f1 > f0; base += 32) {
    const int32_t k = base + lane;
    int32_t nb = 0;
    if (k < a.n_k) {
      int32_t L, lo;
      dec_unit_keys(a, k * a.n_sub + sl, L, lo, nb);
    }
    int32_t incl = nb;
#pragma unroll
    for (int32_t o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, nb > 0 && run + incl > f0);
    if (m) {
      const int32_t j = __ffs(m) - 1;
      const int32_t incl_j = __shfl_sync(0xffffffffu, incl, j);
      const int32_t nb_j = __shfl_sync(0xffffffffu, nb, j);
      sk = base + j;
      sblk = static_cast<int32_t>(f0 - (run + incl_j - nb_j));
      found = true;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    cur[0] = sk;
    cur[1] = sblk;
    cur[2] = found ? static_cast<int32_t>(f1 - f0) : 0;
    cur[3] = sl;
    cur[4] = static_cast<int32_t>(T);
    cur[5] = static_cast<int32_t>(f0);
  }
}

// One arrival on a cut unit's ticket for this call; true for the arrival that
// completes n (this CTA is then the last to finish the unit).  A word left by
// another call starts over at 1.  The compare-and-swap retries only when
// another CTA of the unit arrived in between, so n - 1 retries at most; the
// bound is a safeguard.
__device__ __forceinline__ bool dec_ticket_arrive(unsigned long long *t, unsigned long long epoch,
                                                  uint32_t n) {
  unsigned long long cur = atomicAdd(t, 0ull);
  for (int32_t i = 0; i < 1024; ++i) {
    const unsigned long long want = (cur >> 16) == epoch ? cur + 1ull : (epoch << 16) | 1ull;
    const unsigned long long prev = atomicCAS(t, cur, want);
    if (prev == cur) return static_cast<uint32_t>(want & 0xFFFFull) == n;
    cur = prev;
  }
  status_record(1u, 0xFDu, 8);
  return false;
}

// Shared memory of the decode kernel.  bf16 cache: four K/V stages the TMA
// fills directly.  FP8 cache: two staging slots of raw E4M3 rows (TMA; half the
// bytes of a bf16 block each) and three fp16 K/V stages the conversion warps
// fill for the MMA (block j+1 is converted while block j is multiplied).
template <bool F8>
struct DecLayoutT {
  static constexpr int32_t S = F8 ? 3 : kDecStages;   // K/V stages the MMA reads
  static constexpr int32_t S8 = F8 ? 2 : 0;           // FP8 staging slots
  static constexpr uint32_t kKBox = kDecBN * kRowBytes;    // 64 keys x 64 dims: 8 KB
  static constexpr uint32_t kQOff = 0;                     // 128 rows x 3 boxes: 48 KB
  static constexpr uint32_t kKVOff = kQStageBytes;
  static constexpr uint32_t kKVStage = 5 * kKBox;          // K: 3 boxes, V: 2 boxes
  static constexpr uint32_t kK8 = kDecBN * kDqk;           // 64 keys x 192 E4M3: 12 KB
  static constexpr uint32_t kStg = kK8 + kDecBN * kDv;     // + 64 x 128 E4M3: 20 KB
  static constexpr uint32_t kStgOff = kKVOff + S * kKVStage;
  static constexpr uint32_t kBarOff = kStgOff + S8 * kStg;
  // q_full q_ready q_empty | kv_full[S] k_ready[S] kv_empty[S] | s_full[2] p_full[2] pv_done
  // o_empty drain | stg_full[S8] stg_empty[S8] | q_tmem1 part_out last_known q_tfree[2]
  // (bar 1 is q_tmem0: a query tile rotated and in TMEM buffer 0)
  static constexpr uint32_t kNumBars = 3 + 3 * S + 7 + 2 * S8 + 6;  // + q_rot
  // tmem slot, abort flag, cursor[6], the "last to finish a cut unit" flag
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kTurnsOff = (kMiscOff + 40 + 7) & ~7u;
  static constexpr uint32_t kBytes = kTurnsOff + 32 * 8;
  static constexpr uint32_t kDynSmem = kBytes + 1024;
};
using DecLayout = DecLayoutT<false>;
static_assert(DecLayoutT<false>::kDynSmem <= 232448, "decode kernel shared memory");
static_assert(DecLayoutT<true>::kDynSmem <= 232448, "decode kernel shared memory (FP8)");

// ---------------------------------------------------------------- FP8 cache
// Two E4M3 values (the low byte first) -> f16x2; exact (E4M3 is a subset of f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t d;
  const uint16_t v = static_cast<uint16_t>(two);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
  return d;
}
__device__ __forceinline__ uint4 e4m3x8_to_f16(uint2 v) {
  return make_uint4(e4m3x2_to_f16x2(v.x & 0xffffu), e4m3x2_to_f16x2(v.x >> 16),
                    e4m3x2_to_f16x2(v.y & 0xffffu), e4m3x2_to_f16x2(v.y >> 16));
}
__device__ __forceinline__ float f16lo(uint32_t w) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(w));
  return f;
}
__device__ __forceinline__ float f16hi(uint32_t w) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(w));
  return f;
}
// Element e (0..7) of an 8 x f16 chunk held as four words.
__device__ __forceinline__ float f16_at(const uint32_t (&w)[4], int e) {
  return (e & 1) ? f16hi(w[e >> 1]) : f16lo(w[e >> 1]);
}

// One FP8 K/V block of 64 keys (staging: 64 rows of 192 E4M3 K values, then 64
// rows of 128 E4M3 V values) -> the fp16 stage the MMA reads, in the layout the
// TMA gives a bf16 block (K in 3 boxes, V in 2, 128-byte rows, 128-byte
// swizzle): RoPE on K dims 0..63 at positions kp + row, V rows outside [r0, r1)
// (keys no query sees) written as zeros.  nthr threads.
__device__ void dec_convert_fp8(const uint8_t *stg, uint8_t *kv, int32_t kp, int32_t r0, int32_t r1,
                                bool rope_on, int32_t style, const unsigned long long *turns,
                                int32_t tid, int32_t nthr) {
  constexpr uint32_t kBox = kDecBN * kRowBytes;
  constexpr uint32_t kK8 = kDecBN * kDqk;
  // K dims 64..191 (boxes 1, 2), then V (boxes 3, 4): 16 chunks of 8 values a
  // row each, in two loops so that no warp splits between K and V
#pragma unroll 2
  for (int32_t u = tid; u < kDecBN * 16; u += nthr) {
    const int32_t r = u >> 4, c = u & 15;
    const uint2 v = *reinterpret_cast<const uint2 *>(stg + r * kDqk + 64 + c * 8);
    *swz_chunk(kv + (1 + (c >> 3)) * kBox, r, c & 7) = e4m3x8_to_f16(v);
  }
#pragma unroll 2
  for (int32_t u = tid; u < kDecBN * 16; u += nthr) {
    const int32_t r = u >> 4, c = u & 15;
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (r >= r0 && r < r1) o = e4m3x8_to_f16(*reinterpret_cast<const uint2 *>(stg + kK8 + r * kDv + c * 8));
    *swz_chunk(kv + (3 + (c >> 3)) * kBox, r, c & 7) = o;
  }
  // K dims 0..63 (box 0), rotated
  if (!rope_on || style == 0) {
    for (int32_t u = tid; u < kDecBN * 8; u += nthr) {
      const int32_t r = u >> 3, c = u & 7;
      const uint4 v4 = e4m3x8_to_f16(*reinterpret_cast<const uint2 *>(stg + r * kDqk + c * 8));
      uint32_t w[4] = {v4.x, v4.y, v4.z, v4.w};
      if (rope_on) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float cs, sn;
          rope_cs(kp + r, turns[4 * c + e], cs, sn);
          const float x = f16lo(w[e]), y = f16hi(w[e]);
          w[e] = pack_f16x2(x * cs - y * sn, x * sn + y * cs);
        }
      }
      *swz_chunk(kv, r, c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    // pairs (t, t+32): chunk c (dims 8c..8c+7) with chunk c + 4
    for (int32_t u = tid; u < kDecBN * 4; u += nthr) {
      const int32_t r = u >> 2, c = u & 3;
      const uint4 a4 = e4m3x8_to_f16(*reinterpret_cast<const uint2 *>(stg + r * kDqk + c * 8));
      const uint4 b4 = e4m3x8_to_f16(*reinterpret_cast<const uint2 *>(stg + r * kDqk + (c + 4) * 8));
      const uint32_t a[4] = {a4.x, a4.y, a4.z, a4.w}, b[4] = {b4.x, b4.y, b4.z, b4.w};
      uint32_t oa[4], ob[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        float cs0, sn0, cs1, sn1;
        rope_cs(kp + r, turns[8 * c + e], cs0, sn0);
        rope_cs(kp + r, turns[8 * c + e + 1], cs1, sn1);
        const float x0 = f16_at(a, e), y0 = f16_at(b, e), x1 = f16_at(a, e + 1), y1 = f16_at(b, e + 1);
        oa[e >> 1] = pack_f16x2(x0 * cs0 - y0 * sn0, x1 * cs1 - y1 * sn1);
        ob[e >> 1] = pack_f16x2(x0 * sn0 + y0 * cs0, x1 * sn1 + y1 * cs1);
      }
      *swz_chunk(kv, r, c) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
      *swz_chunk(kv, r, c + 4) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    }
  }
}

// The raw E4M3 block of a staging slot, held in registers between the two
// halves of the conversion: 64 keys x (192 + 128) bytes = 1280 16-byte units,
// kFp8Per per thread for NTHR threads.  Unit order: K dims 0..63 (box 0, the
// rotated ones) first, then K dims 64..191, then V, so that each of a thread's
// units is of one kind across the whole warp.
constexpr int32_t kFp8UnitsK0 = kDecBN * 4;    // K dims 0..63: 4 units of 16 a row
constexpr int32_t kFp8UnitsK = kDecBN * 12;    // all of K
constexpr int32_t kFp8Units = kDecBN * 20;     // K and V
template <int32_t NTHR>
struct Fp8Regs {
  static constexpr int32_t kPer = kFp8Units / NTHR;
  static_assert(kFp8Units % NTHR == 0 && kFp8UnitsK0 % NTHR == 0 && kFp8UnitsK % NTHR == 0,
                "each unit index of a thread has one kind");
  uint4 raw[kPer];
};

// Row, first dim and staging offset of unit u.
__device__ __forceinline__ void fp8_unit(int32_t u, int32_t &r, int32_t &c16, uint32_t &off) {
  constexpr uint32_t kK8 = kDecBN * kDqk;
  if (u < kFp8UnitsK0) {
    r = u >> 2;
    c16 = u & 3;
    off = r * kDqk + c16 * 16;
  } else if (u < kFp8UnitsK) {
    const int32_t v = u - kFp8UnitsK0;
    r = v >> 3;
    c16 = 4 + (v & 7);
    off = r * kDqk + c16 * 16;
  } else {
    const int32_t v = u - kFp8UnitsK;
    r = v >> 3;
    c16 = v & 7;
    off = kK8 + r * kDv + c16 * 16;
  }
}

// First half: the staging slot's bytes into registers (all loads in flight
// together).  The slot may be refilled as soon as this returns.
template <int32_t NTHR>
__device__ __forceinline__ void fp8_load(const uint8_t *stg, Fp8Regs<NTHR> &x, int32_t tid) {
#pragma unroll
  for (int32_t i = 0; i < Fp8Regs<NTHR>::kPer; ++i) {
    int32_t r, c16;
    uint32_t off;
    fp8_unit(tid + i * NTHR, r, c16, off);
    x.raw[i] = *reinterpret_cast<const uint4 *>(stg + off);
  }
}

// Second half: convert to fp16 (exact) into the stage the MMA reads, in the
// layout the TMA gives a bf16 block (K in 3 boxes, V in 2, 128-byte rows,
// 128-byte swizzle); with rotate, K dims 0..63 are rotated at positions kp + row
// (pairs (2t, 2t+1)); V rows outside [r0, r1) (keys no query sees) become zeros.
template <int32_t NTHR>
__device__ __forceinline__ void fp8_store(uint8_t *kv, const Fp8Regs<NTHR> &x, int32_t kp, int32_t r0,
                                          int32_t r1, bool rotate, const unsigned long long *turns,
                                          int32_t tid) {
  constexpr uint32_t kBox = kDecBN * kRowBytes;
#pragma unroll
  for (int32_t i = 0; i < Fp8Regs<NTHR>::kPer; ++i) {
    const int32_t u = tid + i * NTHR;
    int32_t r, c16;
    uint32_t off;
    fp8_unit(u, r, c16, off);
    const uint4 v = x.raw[i];
    uint4 lo = e4m3x8_to_f16(make_uint2(v.x, v.y));
    uint4 hi = e4m3x8_to_f16(make_uint2(v.z, v.w));
    int32_t bi;  // box index in the stage
    if (i * NTHR < kFp8UnitsK) {
      bi = c16 >> 2;
      if (i * NTHR < kFp8UnitsK0 && rotate) {
        // pairs 8 c16 .. 8 c16 + 7, one per 32-bit word
        uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int32_t e = 0; e < 8; ++e) {
          float cs, sn;
          rope_cs(kp + r, turns[8 * c16 + e], cs, sn);
          const float a = f16lo(w[e]), b = f16hi(w[e]);
          w[e] = pack_f16x2(a * cs - b * sn, a * sn + b * cs);
        }
        lo = make_uint4(w[0], w[1], w[2], w[3]);
        hi = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else {
      bi = 3 + (c16 >> 2);
      if (r < r0 || r >= r1) lo = hi = make_uint4(0u, 0u, 0u, 0u);
    }
    // The eight threads of a quarter warp store one row into two boxes (K dims
    // 64..191, V) or two rows into one box (K dims 0..63).  Boxes are 8 KB apart
    // and so share banks: threads of an odd box store their two 16-byte halves
    // in the other order, so one store instruction writes the even chunks of one
    // box and the odd chunks of the other (rows next to each other already
    // differ in their swizzle parity).
    uint8_t *box = kv + bi * kBox;
    const int32_t ch = (c16 & 3) * 2;
    const bool swap = bi & 1;
    *swz_chunk(box, r, ch + (swap ? 1 : 0)) = swap ? hi : lo;
    *swz_chunk(box, r, ch + (swap ? 0 : 1)) = swap ? lo : hi;
  }
}

// The Q tile's rows [0, R) to fp16 in place: boxes 1 and 2, and box 0 unless
// the RoPE pass has already written it as fp16.  nthr threads.
__device__ void dec_q_to_f16(uint8_t *q, int32_t R, bool box0, int32_t tid, int32_t nthr) {
  const int32_t first = box0 ? 0 : 1;
  const int32_t nch = (3 - first) * 8;
  for (int32_t u = tid; u < R * nch; u += nthr) {
    const int32_t r = u / nch, c = u % nch + first * 8;
    uint4 *p = reinterpret_cast<uint4 *>(q + (c >> 3) * kQBoxBytes + r * kRowBytes + (c & 7) * 16);
    const uint4 v = *p;
    *p = make_uint4(pack_f16x2(bf16lo(v.x), bf16hi(v.x)), pack_f16x2(bf16lo(v.y), bf16hi(v.y)),
                    pack_f16x2(bf16lo(v.z), bf16hi(v.z)), pack_f16x2(bf16lo(v.w), bf16hi(v.w)));
  }
}

// Threads: 384 (bf16 cache) or 512 (FP8 cache: warps 12-15 join the
// conversion of the cache blocks).
template <bool F8>
struct DecThreads {
  static constexpr int32_t kAll = F8 ? 512 : kThreads;
  static constexpr int32_t kConv = kAll - 256;  // warps 8.. : RoPE / conversion
};

template <bool F8>
__global__ void __launch_bounds__(DecThreads<F8>::kAll, 1)
    sinkattn_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ DecArgs args) {
  using Ly = DecLayoutT<F8>;
  constexpr int32_t S = Ly::S;
  constexpr int32_t S8 = Ly::S8;
  constexpr int32_t BN = kDecBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int32_t warp = threadIdx.x >> 5;
  const int32_t lane = threadIdx.x & 31;

  auto bar = [&](uint32_t i) { return sbase + Ly::kBarOff + i * 8; };
  const uint32_t B_QFULL = bar(0), B_QEMPTY = bar(2);
  auto B_KVFULL = [&](uint32_t s) { return bar(3 + s); };
  auto B_KREADY = [&](uint32_t s) { return bar(3 + S + s); };
  auto B_KVEMPTY = [&](uint32_t s) { return bar(3 + 2 * S + s); };
  auto B_SFULL = [&](uint32_t b) { return bar(3 + 3 * S + b); };
  auto B_PFULL = [&](uint32_t b) { return bar(3 + 3 * S + 2 + b); };
  const uint32_t B_PVDONE = bar(3 + 3 * S + 4);
  const uint32_t B_OEMPTY = bar(3 + 3 * S + 5);
  const uint32_t B_DRAIN = bar(3 + 3 * S + 6);
  auto B_STGFULL = [&](uint32_t s8) { return bar(3 + 3 * S + 7 + s8); };
  auto B_STGEMPTY = [&](uint32_t s8) { return bar(3 + 3 * S + 7 + S8 + s8); };
  // a query tile rotated and in TMEM buffer b (the conversion threads); buffer
  // b free again (a commit after the last QK^T that read it)
  auto B_QTMEM = [&](uint32_t b) { return b ? bar(3 + 3 * S + 7 + 2 * S8) : bar(1); };
  auto B_QTFREE = [&](uint32_t b) { return bar(3 + 3 * S + 7 + 2 * S8 + 3 + b); };
  const uint32_t B_QROT = bar(3 + 3 * S + 7 + 2 * S8 + 5);  // the tile rotated (all conversion threads)
  // a cut unit's partial is out (128 softmax threads), the ticket's answer is known (1)
  const uint32_t B_PARTOUT = bar(3 + 3 * S + 7 + 2 * S8 + 1);
  const uint32_t B_LASTKNOWN = bar(3 + 3 * S + 7 + 2 * S8 + 2);

  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  int32_t *cur_smem = reinterpret_cast<int32_t *>(smem + Ly::kMiscOff + 8);
  volatile int32_t *last_flag = reinterpret_cast<volatile int32_t *>(smem + Ly::kMiscOff + 32);
  unsigned long long *turns = reinterpret_cast<unsigned long long *>(smem + Ly::kTurnsOff);

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    mbar_init(B_QFULL, 1);
    mbar_init(B_QEMPTY, DecThreads<F8>::kConv);  // the conversion threads, once Q is in TMEM
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(B_QTMEM(b), DecThreads<F8>::kConv);
      mbar_init(B_QTFREE(b), 1);
    }
    mbar_init(B_QROT, DecThreads<F8>::kConv);
    mbar_init(B_PARTOUT, 128);
    mbar_init(B_LASTKNOWN, 1);
    for (uint32_t s = 0; s < S; ++s) {
      mbar_init(B_KVFULL(s), 1);
      mbar_init(B_KREADY(s), DecThreads<F8>::kConv);
      mbar_init(B_KVEMPTY(s), 1);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(B_SFULL(b), 1);
      mbar_init(B_PFULL(b), 128);
    }
    mbar_init(B_PVDONE, 1);
    mbar_init(B_OEMPTY, 128);
    mbar_init(B_DRAIN, 1);
    if constexpr (F8) {
      for (uint32_t s8 = 0; s8 < static_cast<uint32_t>(S8); ++s8) {
        mbar_init(B_STGFULL(s8), 1);
        mbar_init(B_STGEMPTY(s8), DecThreads<F8>::kConv);
      }
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) turns[threadIdx.x] = args.rope_turns[threadIdx.x];
  if (warp == 2) {
    tmem_alloc(sbase + Ly::kMiscOff, kDecTmemCols);
    tmem_relinquish();
  }
  if (warp == 3) dec_locate(args, lane, cur_smem);
  // The Q tile has T * G rows; the MMA reads all 128, so the rest stay zero.
  for (uint32_t i = threadIdx.x; i < kQStageBytes / 16; i += DecThreads<F8>::kAll)
    reinterpret_cast<uint4 *>(smem + Ly::kQOff)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int32_t G = args.G;
  const int32_t R = args.R;
  DecCursor c0;
  c0.k = cur_smem[0];
  c0.blk = cur_smem[1];
  c0.left = cur_smem[2];
  c0.s = cur_smem[3];
  c0.first = 1;

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t gq = 0, gk = 0;
      bool ok = true;
      DecCursor c = c0;
      DecSeg sg;
      while (ok && dec_next(c, args, sg)) {
        if (!(ok = wait_bar(B_QEMPTY, (gq & 1) ^ 1, abort_flag, 1))) break;
        mbar_arrive_expect_tx(B_QFULL, args.q_tx_bytes);
#pragma unroll
        for (int cc = 0; cc < 3; ++cc)
          tma_load_3d(sbase + Ly::kQOff + cc * kQBoxBytes, &tm_q, cc * 64, sg.kvh * G, sg.b * args.T,
                      B_QFULL);
        ++gq;
        const int32_t kpos0 = sg.lo + sg.blk0 * BN;
        const int32_t krow0 = sg.b * args.S_cap + kpos0;
        for (int32_t j = 0; j < sg.nblk; ++j) {
          if constexpr (F8) {
            // raw E4M3 rows into a staging slot; the conversion warps fill the MMA's stage
            const uint32_t s8 = gk % S8;
            if (!(ok = wait_bar(B_STGEMPTY(s8), ((gk / S8) & 1) ^ 1, abort_flag, 2))) break;
            mbar_arrive_expect_tx(B_STGFULL(s8), Ly::kStg);
            const uint32_t dst = sbase + Ly::kStgOff + s8 * Ly::kStg;
            tma_load_3d(dst, &tm_k, 0, sg.kvh, krow0 + j * BN, B_STGFULL(s8));
            tma_load_3d(dst + Ly::kK8, &tm_v, 0, sg.kvh, krow0 + j * BN, B_STGFULL(s8));
            ++gk;
            continue;
          }
          const uint32_t st = gk % S;
          if (!(ok = wait_bar(B_KVEMPTY(st), ((gk / S) & 1) ^ 1, abort_flag, 2))) break;
          mbar_arrive_expect_tx(B_KVFULL(st), Ly::kKVStage);
          const uint32_t dst = sbase + Ly::kKVOff + st * Ly::kKVStage;
          if (!args.kv_ring) {
#pragma unroll
            for (int cc = 0; cc < 3; ++cc)
              tma_load_3d(dst + cc * Ly::kKBox, &tm_k, cc * 64, sg.kvh, krow0 + j * BN, B_KVFULL(st));
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
              tma_load_3d(dst + (3 + cc) * Ly::kKBox, &tm_v, cc * 64, sg.kvh, krow0 + j * BN,
                          B_KVFULL(st));
          } else {
            // four 16-key pieces (the maps' boxes are 16 rows), each at its slot
#pragma unroll 1
            for (int32_t pc = 0; pc < BN; pc += 16) {
              const int32_t row = sg.b * args.S_cap + (kpos0 + j * BN + pc) % args.S_cap;
#pragma unroll
              for (int cc = 0; cc < 3; ++cc)
                tma_load_3d(dst + cc * Ly::kKBox + pc * kRowBytes, &tm_k, cc * 64, sg.kvh, row,
                            B_KVFULL(st));
#pragma unroll
              for (int cc = 0; cc < 2; ++cc)
                tma_load_3d(dst + (3 + cc) * Ly::kKBox + pc * kRowBytes, &tm_v, cc * 64, sg.kvh, row,
                            B_KVFULL(st));
            }
          }
          ++gk;
        }
      }
      if (gq > 0) drain_wait(B_QFULL, (gq - 1) & 1);
      if constexpr (F8) {
        for (uint32_t s8 = 0; s8 < static_cast<uint32_t>(S8); ++s8)
          if (gk > s8) drain_wait(B_STGFULL(s8), ((gk - 1 - s8) / S8) & 1);
      } else {
        for (uint32_t s = 0; s < S; ++s)
          if (gk > s) drain_wait(B_KVFULL(s), ((gk - 1 - s) / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      // dims 0..63 of Q and K are fp16 once rotated here; keys a bf16 cache
      // already holds rotated stay bf16, and Q's rotated dims are bf16 to match
      const uint32_t rot = (args.rope_on && !args.k_rotated) ? 0u : 1u;
      // FP8 cache: every operand (Q, the converted K and V, P) is fp16
      const uint32_t kIdQK = idesc_f32acc(128, BN, F8 ? 0 : 1, 0, 0);
      const uint32_t kIdQKRot = idesc_f32acc(128, BN, F8 ? 0 : rot, 0, 0);
      constexpr uint32_t kIdPV = idesc_f32acc(128, kDv, F8 ? 0 : 1, 0, 1);
      constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
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
      DecCursor c = c0;
      DecSeg sg;
      while (ok && dec_next(c, args, sg)) {
        const uint32_t qb = gq & 1;
        if (!(ok = wait_bar(B_QTMEM(qb), (gq >> 1) & 1, abort_flag, 3))) break;
        tc_fence_after();
        for (int32_t j = 0; ok && j < sg.nblk; ++j) {
          const uint32_t st = (gk + j) % S;
          // QK^T(j) goes out before PV(j-1) waits for the softmax of block
          // j-1, so the two overlap.  The stage block j needs was last read by
          // PV(j-S), issued in an earlier pass of this loop.
          if (!(ok = wait_bar(B_KREADY(st), ((gk + j) / S) & 1, abort_flag, 6))) break;
          tc_fence_after();
          const uint32_t s_t = tmem + ((gs + j) & 1) * BN;
#pragma unroll
          for (int kstep = 0; kstep < kDqk / 16; ++kstep) {
            const uint32_t box = kstep >> 2, off = (kstep & 3) * 32;
            mma_ts2(s_t, tmem + dec_tmem_q(qb) + kstep * 8,
                    kv_lo + st * kStageLo + ((box * Ly::kKBox + off) >> 4), kDescHi,
                    box == 0 ? kIdQKRot : kIdQK, kstep > 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit(B_SFULL((gs + j) & 1));
          if (j == sg.nblk - 1) mma_commit(B_QTFREE(qb));  // the unit's last read of its tile
          if (j > 0 && !(ok = issue_pv(gs + j - 1, (gk + j - 1) % S, j == 1))) break;
        }
        if (ok) ok = issue_pv(gs + sg.nblk - 1, (gk + sg.nblk - 1) % S, sg.nblk == 1);
        ++gq;
        gk += sg.nblk;
        gs += sg.nblk;
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
    const int32_t W = args.window;
    uint32_t gs = 0, gpv = 0, gcut = 0;
    bool ok = true;
    DecCursor c = c0;
    DecSeg sg;
    // the list's CTAs, its total blocks, and the flat index of this CTA's next block
    const int32_t n_grp = static_cast<int32_t>(gridDim.x) / args.n_sub;
    const int64_t Tb = cur_smem[4];
    int64_t flat = cur_smem[5];
    while (ok && dec_next(c, args, sg)) {
      const int64_t F0 = flat - sg.blk0;  // the unit's blocks are [F0, F0 + nblk_u) of the list
      flat += sg.nblk;
      // query t sits at position L - T + t and sees cache keys
      // [max(0, pos - W + 1), pos], here limited to this segment's keys
      const int32_t pos = sg.L - args.T + t;
      const int32_t kfirst = sg.lo + sg.blk0 * BN;
      const int32_t klast = min(kfirst + sg.nblk * BN, sg.L) - 1;
      const bool rvalid = row < R && pos >= 0;
      int32_t qlo = max(kfirst, W > 0 ? pos - W + 1 : 0);
      int32_t qhi = min(pos, klast);
      // no visible key in this segment (or no such row): nothing is visible
      if (!rvalid || qhi < qlo) { qlo = 1 << 30; qhi = 1 << 30; }
      // FP8 cache: the keys' scale folds into the logit scale, the values' into o
      const float sc = args.scale_log2 * (F8 ? __ldg(args.k_scale + sg.kvh) : 1.f);
      float m = -INFINITY, l = 0.f;
      for (int32_t j = 0; ok && j < sg.nblk; ++j) {
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
          const int32_t kb = kfirst + j * BN;
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
            r[k >> 1] = F8 ? pack_f16x2(p.x, p.y) : pack_bf16x2(p.x, p.y);
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
            for (int32_t cb = 0; cb < kDv; cb += 32) {
              uint32_t o[32];
              tmem_ld32p(o_t + cb, o);
              tmem_wait_ld();
              reg_fence<32>(o);
#pragma unroll
              for (int32_t k = 0; k < 32; k += 2) {
                const float2 v = fmul2(make_float2(__uint_as_float(o[k]), __uint_as_float(o[k + 1])),
                                       make_float2(alpha_row, alpha_row));
                o[k] = __float_as_uint(v.x);
                o[k + 1] = __float_as_uint(v.y);
              }
              tmem_st32p(o_t + cb, o);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        mbar_arrive(B_PFULL(buf));
        ++gs;
      }
      if (!ok) break;
      // ---------------- end of the segment
      if (!(ok = wait_bar_warp(B_PVDONE, (gpv + sg.nblk - 1) & 1, abort_flag, 9))) break;
      gpv += sg.nblk;
      tc_fence_after();
      const bool whole_unit = sg.blk0 == 0 && sg.nblk == sg.nblk_u;
      if (warp_active) {
        const uint32_t o_t = tmem + lane_off + kDecTmemO;
        const int32_t head = sg.kvh * G + g;
        // whole unit: eqs. (2)-(3) with the sink added once,
        //   M = max(m, sink), L = l 2^(m - M) + 2^(sink - M), o = O 2^(m - M) / L;
        // else the unnormalised partial (m, l, O) for the merge
        float scale_o = 1.f, lse_v = 0.f;
        if (whole_unit) {
          const float sk2 = __ldg(args.sink + head) * kLog2e;
          const float M = fmaxf(m, sk2);
          if (M == -INFINITY) {
            scale_o = 0.f;
            lse_v = -INFINITY;
          } else {
            const float a1 = m == -INFINITY ? 0.f : ex2(m - M);
            const float a2 = sk2 == -INFINITY ? 0.f : ex2(sk2 - M);
            const float Lw = l * a1 + a2;
            scale_o = a1 / Lw;
            lse_v = (M + __log2f(Lw)) * kLn2;
          }
        }
        // FP8 cache: the values' scale multiplies O (partials included: the
        // merge is linear in O)
        const float vs = F8 ? __ldg(args.v_scale + sg.kvh) : 1.f;
        scale_o *= vs;
        const size_t orow = (static_cast<size_t>(sg.b) * args.T + t) * args.Hq + head;
        const size_t prow = (static_cast<size_t>(blockIdx.x) * 2 + (sg.first ? 0 : 1)) * R + row;
        const bool st_ok = row < R && (whole_unit ? SA_OUT(orow, args.n_rows, 0x21)
                                                  : SA_IN(prow, args.n_part_rows, 0x22));
#pragma unroll 1
        for (int32_t cb = 0; cb < kDv; cb += 32) {
          uint32_t o[32];
          tmem_ld32p(o_t + cb, o);
          tmem_wait_ld();
          reg_fence<32>(o);
          if (st_ok) {
            if (whole_unit) {
              uint4 *dst = reinterpret_cast<uint4 *>(args.out + orow * kDv + cb);
#pragma unroll
              for (int32_t q4 = 0; q4 < 4; ++q4) {
                uint32_t w4[4];
#pragma unroll
                for (int32_t e = 0; e < 4; ++e)
                  w4[e] = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2 * e]) * scale_o,
                                      __uint_as_float(o[q4 * 8 + 2 * e + 1]) * scale_o);
                dst[q4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
              }
            } else {
              float4 *dst = reinterpret_cast<float4 *>(args.part_o + prow * kDv + cb);
#pragma unroll
              for (int32_t q4 = 0; q4 < 8; ++q4)
                dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * vs, __uint_as_float(o[4 * q4 + 1]) * vs,
                                      __uint_as_float(o[4 * q4 + 2]) * vs, __uint_as_float(o[4 * q4 + 3]) * vs);
            }
          }
        }
        if (st_ok) {
          if (whole_unit)
            args.lse[orow] = lse_v;
          else
            reinterpret_cast<float4 *>(args.part_ml)[prow] = make_float4(m, l, 0.f, 0.f);
        }
      }
      tc_fence_before();
      mbar_arrive(B_OEMPTY);
      if (!whole_unit) {
        // A cut unit: this CTA's partial is out; the CTA that completes the
        // unit's ticket merges every partial of the unit (they are written
        // before their CTA's arrival, which the fences order device-wide).
        // Group i of the list holds blocks [Tb i / n_grp, Tb (i + 1) / n_grp).
        const int64_t F1 = F0 + sg.nblk_u;
        auto grp_of = [&](int64_t f) { return static_cast<int32_t>(((f + 1) * n_grp - 1) / Tb); };
        auto has_part = [&](int32_t i) { return Tb * i / n_grp != Tb * (i + 1) / n_grp; };
        const int32_t c_first = grp_of(F0), c_last = grp_of(F1 - 1);
        uint32_t n_part = 0;
        for (int32_t i = c_first; i <= c_last; ++i) n_part += has_part(i) ? 1u : 0u;
        __threadfence();
        mbar_arrive(B_PARTOUT);
        if (threadIdx.x == 128) {
          // (no early exit here: the whole warp meets again in the wait below;
          // an aborted CTA merges nothing)
          const bool all_out = wait_bar(B_PARTOUT, gcut & 1, abort_flag, 14);
          *last_flag = all_out && SA_IN(sg.u, args.n_units, 0x23) &&
                               dec_ticket_arrive(args.tickets + sg.u, args.epoch, n_part)
                           ? 1 : 0;
          mbar_arrive(B_LASTKNOWN);
        }
        if (!(ok = wait_bar_warp(B_LASTKNOWN, gcut & 1, abort_flag, 15))) break;
        ++gcut;
        if (*last_flag) {
          __threadfence();
          // M = max(sink, m_i), L = 2^(sink - M) + sum_i l_i 2^(m_i - M),
          // o = sum_i 2^(m_i - M) O_i / L, in group order (eq. (2) over the
          // partition of the unit's keys, the sink once).  All 128 threads:
          // item (row r, 32 dims), four a row; each item's loads go out
          // together.
          const int32_t sl = static_cast<int32_t>(blockIdx.x) % args.n_sub;
          const float4 *ml = reinterpret_cast<const float4 *>(args.part_ml);
          for (int32_t wi = row; wi < R * 4; wi += 128) {
            const int32_t r = wi >> 2, cb = (wi & 3) * 32;
            const int32_t head = sg.kvh * G + r % G;
            const size_t orow = (static_cast<size_t>(sg.b) * args.T + r / G) * args.Hq + head;
            auto prow_of = [&](int32_t i) {
              const size_t cta = static_cast<size_t>(i) * args.n_sub + sl;
              return (cta * 2 + ((i == c_first && Tb * i / n_grp < F0) ? 1 : 0)) * R + r;
            };
            if (!SA_OUT(orow, args.n_rows, 0x24)) continue;
            // (checking builds: every partial row the merge reads is in the buffer)
            if (!(SA_IN(prow_of(c_first), args.n_part_rows, 0x25) &&
                  SA_IN(prow_of(c_last), args.n_part_rows, 0x25)))
              continue;
            const float sk_raw = __ldg(args.sink + head);
            const float sk2 = sk_raw == -INFINITY ? -INFINITY : sk_raw * kLog2e;
            float M = sk2;
#pragma unroll 4
            for (int32_t i = c_first; i <= c_last; ++i)
              if (has_part(i)) M = fmaxf(M, __ldcg(ml + prow_of(i)).x);
            uint4 *dst = reinterpret_cast<uint4 *>(args.out + orow * kDv + cb);
            if (M == -INFINITY) {
#pragma unroll
              for (int32_t q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(0u, 0u, 0u, 0u);
              if (cb == 0) args.lse[orow] = -INFINITY;
              continue;
            }
            float Ls = sk2 == -INFINITY ? 0.f : ex2(sk2 - M);
            float acc[32];
#pragma unroll
            for (int32_t e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll 2
            for (int32_t i = c_first; i <= c_last; ++i) {
              if (!has_part(i)) continue;
              const size_t pr = prow_of(i);
              const float4 *src = reinterpret_cast<const float4 *>(args.part_o + pr * kDv + cb);
              float4 o4[8];
#pragma unroll
              for (int32_t q4 = 0; q4 < 8; ++q4) o4[q4] = __ldcg(src + q4);
              const float4 v = __ldcg(ml + pr);
              const float w = v.x == -INFINITY ? 0.f : ex2(v.x - M);
              Ls += v.y * w;
#pragma unroll
              for (int32_t q4 = 0; q4 < 8; ++q4) {
                acc[4 * q4] += w * o4[q4].x;
                acc[4 * q4 + 1] += w * o4[q4].y;
                acc[4 * q4 + 2] += w * o4[q4].z;
                acc[4 * q4 + 3] += w * o4[q4].w;
              }
            }
#pragma unroll
            for (int32_t q4 = 0; q4 < 4; ++q4)
              dst[q4] = make_uint4(pack_bf16x2(acc[8 * q4] / Ls, acc[8 * q4 + 1] / Ls),
                                   pack_bf16x2(acc[8 * q4 + 2] / Ls, acc[8 * q4 + 3] / Ls),
                                   pack_bf16x2(acc[8 * q4 + 4] / Ls, acc[8 * q4 + 5] / Ls),
                                   pack_bf16x2(acc[8 * q4 + 6] / Ls, acc[8 * q4 + 7] / Ls));
            if (cb == 0) args.lse[orow] = (M + __log2f(Ls)) * kLn2;
          }
        }
      }
    }
  } else if (warp >= 8) {
    // ============================================================ RoPE
    const int32_t tid = threadIdx.x - 256;
    uint32_t gq = 0, gk = 0;
    bool ok = true;
    DecCursor c = c0;
    DecSeg sg;
    while (ok && dec_next(c, args, sg)) {
      if (!(ok = wait_bar_warp(B_QFULL, gq & 1, abort_flag, 10))) break;
      if (args.rope_on && tid < 128) {
        if (!F8 && args.k_rotated)
          rope_q_tile<true>(smem + Ly::kQOff, G, args.T, sg.L - args.T, args.rope_style, turns, tid);
        else
          rope_q_tile(smem + Ly::kQOff, G, args.T, sg.L - args.T, args.rope_style, turns, tid);
      }
      if constexpr (F8) {
        // every MMA operand is fp16 with an FP8 cache (the rotation above
        // already wrote box 0 as fp16; the conversion touches the other boxes)
        dec_q_to_f16(smem + Ly::kQOff, R, !args.rope_on, tid, DecThreads<F8>::kConv);
      }
      // every conversion thread's rotation / conversion of the tile is done
      // before any thread copies rows of it
      mbar_arrive(B_QROT);
      if (!(ok = wait_bar_warp(B_QROT, gq & 1, abort_flag, 13))) break;
      // TMEM buffer qb is free once the last QK^T of the unit two back read it
      const uint32_t qb = gq & 1;
      if (!(ok = wait_bar_warp(B_QTFREE(qb), ((gq >> 1) & 1) ^ 1, abort_flag, 14))) break;
      tc_fence_after();
      {
        // one row a thread (lane quarter warp % 4); with an FP8 cache warps
        // 8-11 copy boxes 0 and 1 and warps 12-15 box 2
        const int32_t q4 = warp & 3, row = q4 * 32 + lane;
        const int32_t b0 = (F8 && warp >= 12) ? 2 : 0, b1 = (F8 && warp < 12) ? 2 : 3;
        if (q4 * 32 < R) {
          const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + dec_tmem_q(qb);
#pragma unroll 1
          for (int32_t b = b0; b < b1; ++b) {
            uint32_t w[32];
#pragma unroll
            for (int32_t ch = 0; ch < 8; ++ch) {
              const uint4 v = *swz_chunk(smem + Ly::kQOff + b * kQBoxBytes, row, ch);
              w[4 * ch] = v.x;
              w[4 * ch + 1] = v.y;
              w[4 * ch + 2] = v.z;
              w[4 * ch + 3] = v.w;
            }
            tmem_st32p(taddr + b * 32, w);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(B_QTMEM(qb));
      mbar_arrive(B_QEMPTY);
      ++gq;
      const int32_t kpos0 = sg.lo + sg.blk0 * BN;
      // keys no query of the unit can see: below the window or past the cache
      const int32_t vis_lo = args.window > 0 ? max(0, sg.L - args.T - args.window + 1) : 0;
      for (int32_t j = 0; j < sg.nblk; ++j) {
        const uint32_t st = gk % S;
        if constexpr (F8) {
          const uint32_t s8 = gk % S8;
          if (!(ok = wait_bar_warp(B_STGFULL(s8), (gk / S8) & 1, abort_flag, 11))) break;
          const int32_t kp = kpos0 + j * BN;
          const int32_t r0 = min(BN, max(0, vis_lo - kp)), r1 = max(r0, min(BN, sg.L - kp));
          const bool rotate = args.rope_on && !args.k_rotated;
          uint8_t *stage = smem + Ly::kKVOff + st * Ly::kKVStage;
          if (!rotate || args.rope_style == 0) {
            // the raw block into registers, the staging slot back to the TMA
            // at once, then the wait for the fp16 stage
            Fp8Regs<DecThreads<F8>::kConv> x;
            fp8_load(smem + Ly::kStgOff + s8 * Ly::kStg, x, tid);
            mbar_arrive(B_STGEMPTY(s8));
            // the fp16 stage is free once the PV that last read it completed
            if (!(ok = wait_bar_warp(B_KVEMPTY(st), ((gk / S) & 1) ^ 1, abort_flag, 12))) break;
            fp8_store(stage, x, kp, r0, r1, rotate, turns, tid);
          } else {
            if (!(ok = wait_bar_warp(B_KVEMPTY(st), ((gk / S) & 1) ^ 1, abort_flag, 12))) break;
            dec_convert_fp8(smem + Ly::kStgOff + s8 * Ly::kStg, stage, kp, r0, r1, true,
                            args.rope_style, turns, tid, DecThreads<F8>::kConv);
            mbar_arrive(B_STGEMPTY(s8));
          }
          fence_proxy_async_smem();
          mbar_arrive(B_KREADY(st));
          ++gk;
          continue;
        }
        if (!(ok = wait_bar_warp(B_KVFULL(st), (gk / S) & 1, abort_flag, 11))) break;
        uint8_t *kv = smem + Ly::kKVOff + st * Ly::kKVStage;
        const int32_t kp = kpos0 + j * BN;
        if (args.rope_on && !args.k_rotated) rope_k_rows(kv, BN, kp, args.rope_style, turns, tid);
        // Their scores are masked, but P = 0 times a NaN value is NaN: zero
        // the value rows of keys outside [vis_lo, L), whose cache rows (past
        // the sequence, or old ring slots) may hold anything.
        const int32_t r0 = min(BN, max(0, vis_lo - kp)), r1 = max(r0, min(BN, sg.L - kp));
        if (r0 > 0 || r1 < BN) {
          for (int32_t u = tid; u < BN * 16; u += 128) {
            const int32_t r = u >> 4, ch = u & 15;  // row, 16-byte chunk of its 256 bytes
            if (r < r0 || r >= r1)
              *reinterpret_cast<uint4 *>(kv + (3 + (ch >> 3)) * Ly::kKBox + r * kRowBytes +
                                         (ch & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
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
