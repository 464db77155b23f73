// band_kernel.cuh -- sliding-window (SWA) prefill for 8 query heads per KV head.
//
// Computes the attention layer of the MiMo-V2-Flash Technical Report (§2.2
// eqs. (1)-(3), shapes of §2.1 Table 1) for the sliding-window layers: key j
// is visible to query i iff i - W < j <= i, W <= 128.
//
// A tile is 16 consecutive tokens x the 8 query heads of one KV head (128 MMA
// rows, row r = token * 8 + head).  Its keys are the 16-key segments
// [t0 - 128, t0 + 16) (W = 128: 9 segments, 144 keys), so one QK^T MMA of
// N = 144 and one PV of K = 144 cover the whole band of the tile.
//
// Each CTA walks a contiguous run of tiles of one (sequence, KV head) lane at a
// time (the flattened tile list is cut into gridDim.x equal pieces), and keeps
// the keys and values of the band in a shared-memory ring of 12 segments: a
// tile loads only its own 16 new keys, so K and V are read from memory once,
// and the loads run up to three tiles ahead of the MMAs.
//
// Warp roles (512 threads, one CTA per SM):
//   warp 0       TMA producer: Q tile (3 boxes of 64 dims, 2 stages), new K/V segments.
//   warp 1       MMA issuer: S = Q K^T into TMEM (two MMAs when the band wraps
//                around the end of the ring), then O = P V with P read from TMEM.
//   warp 2       TMEM allocator (S0, S1, O).
//   warp 3       set-up: locates this CTA's first tile.
//   warps 4-11   softmax + epilogue, two threads per row (TMEM lane): warps 4-7
//                take band columns 0..71 and output dims 0..63, warps 8-11 band
//                columns 72..143 and output dims 64..127.  Per tile: row max over
//                the band with the sink (eq. (2); partial maxima swapped through
//                shared memory), P = 2^(s*scale*log2e - m) as bf16 into TMEM, then
//                for the previous tile o = O / l with l = 2^(sink - m) + sum P,
//                and the log-sum-exp.
//   warps 12-15  RoPE on dims 0..63 of the Q tile and of each new K segment.
#pragma once
#include "common.cuh"

namespace sa {

constexpr int32_t kBandSeg = 16;   // keys per ring segment = tokens per tile
constexpr int32_t kBandRing = 12;  // segments in the K/V ring
constexpr int32_t kBandMaxWin = 9; // segments of a full window, W <= 128
constexpr int32_t kBandG = 8;      // query heads per KV head
constexpr int32_t kBandThreads = 512;
constexpr int32_t kBandHalf = 72;  // band columns per softmax thread
constexpr uint32_t kBandPCol = 36; // TMEM column of P (bf16 pairs) within an S buffer

struct BandArgs {
  int32_t Hq, Hkv;
  int32_t window;      // 1..128
  int32_t batch;
  int32_t nseg;        // segments of a full window: ceil((window - 1) / 16) + 1
  int32_t rope_on, rope_style;
  float scale_log2;    // logit scale * log2(e), > 0
  int32_t out_v8;      // 1: out is 32-byte aligned (whole-sector stores)
  const int32_t *cu_seqlens;
  const float *sink;
  __nv_bfloat16 *out;
  float *lse;
  int64_t n_rows;       // rows of out and lse: tokens x Hq (checked stores)
  unsigned long long rope_turns[32];
};

// RoPE on dims 0..63 of a band Q tile (16 tokens x 8 heads, rows t * 8 + g),
// 128 threads.  A thread takes one (token, 16-byte chunk) unit and its angles
// once, then all the heads of that token: the loads of the heads' chunks go
// out together before any rotation (the RoPE warps share their schedulers
// with the softmax warps, so a chain of dependent load-rotate-store steps
// per head would run at a fraction of their issue rate).
__device__ __forceinline__ void band_rope_q(uint8_t *box0, int32_t n_tok, int32_t pos0,
                                            int32_t style, const unsigned long long *turns,
                                            int32_t tid) {
  if (style == 0) {
    // interleaved pairs: 16 tokens x 8 chunks (4 pairs each) = 128 units
    const int32_t t = tid >> 3, c = tid & 7;
    if (t >= n_tok) return;
    float cs[4], sn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) rope_cs(pos0 + t, turns[4 * c + e], cs[e], sn[e]);
    uint4 v[kBandG];
#pragma unroll
    for (int32_t g = 0; g < kBandG; ++g) v[g] = *swz_chunk(box0, t * kBandG + g, c);
#pragma unroll
    for (int32_t g = 0; g < kBandG; ++g) {
      uint32_t w[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = bf16lo(w[e]), y = bf16hi(w[e]);
        w[e] = pack_f16x2(x * cs[e] - y * sn[e], x * sn[e] + y * cs[e]);
      }
      *swz_chunk(box0, t * kBandG + g, c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    // half-split pairs (p, p + 32): 16 tokens x 4 chunk pairs = 64 units, each
    // taken by two threads (4 heads each)
    const int32_t u = tid >> 1, t = u >> 2, c = u & 3, g0 = (tid & 1) * (kBandG / 2);
    if (t >= n_tok) return;
    float cs[8], sn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_cs(pos0 + t, turns[8 * c + e], cs[e], sn[e]);
    uint4 va[kBandG / 2], vb[kBandG / 2];
#pragma unroll
    for (int32_t g = 0; g < kBandG / 2; ++g) {
      va[g] = *swz_chunk(box0, t * kBandG + g0 + g, c);
      vb[g] = *swz_chunk(box0, t * kBandG + g0 + g, c + 4);
    }
#pragma unroll
    for (int32_t g = 0; g < kBandG / 2; ++g) {
      uint32_t a[4] = {va[g].x, va[g].y, va[g].z, va[g].w};
      uint32_t b[4] = {vb[g].x, vb[g].y, vb[g].z, vb[g].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x0 = bf16lo(a[e]), y0 = bf16lo(b[e]);
        const float x1 = bf16hi(a[e]), y1 = bf16hi(b[e]);
        const float c0 = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
        a[e] = pack_f16x2(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
        b[e] = pack_f16x2(x0 * s0 + y0 * c0, x1 * s1 + y1 * c1);
      }
      *swz_chunk(box0, t * kBandG + g0 + g, c) = make_uint4(a[0], a[1], a[2], a[3]);
      *swz_chunk(box0, t * kBandG + g0 + g, c + 4) = make_uint4(b[0], b[1], b[2], b[3]);
    }
  }
}

struct BandLayout {
  static constexpr uint32_t kSegBox = kBandSeg * kRowBytes;   // 16 keys x 64 dims: 2 KB
  static constexpr uint32_t kRingBox = kBandRing * kSegBox;   // 24 KB
  static constexpr uint32_t kQOff = 0;                        // 2 stages x 48 KB
  static constexpr uint32_t kKOff = 2 * kQStageBytes;         // 3 ring boxes (dims 0..191)
  static constexpr uint32_t kVOff = kKOff + 3 * kRingBox;     // 2 ring boxes (dims 0..127)
  static constexpr uint32_t kBarOff = kVOff + 2 * kRingBox;
  // q_full[2] q_ready[2] q_empty[2] seg_full[R] seg_ready[R] seg_empty[R]
  // s_full[2] p_full[2] pv_done o_empty drain pair[2][4]
  static constexpr uint32_t kPairBar = 6 + 3 * kBandRing + 7;
  static constexpr uint32_t kNumBars = kPairBar + 8;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;  // tmem, abort, cursor[4]
  static constexpr uint32_t kTurnsOff = (kMiscOff + 32 + 7) & ~7u;
  // partial (max, sum) of each row half, double-buffered by tile parity
  static constexpr uint32_t kXchgOff = kTurnsOff + 32 * 8;
  static constexpr uint32_t kBytes = kXchgOff + 2 * 2 * 128 * 8;
  static constexpr uint32_t kDynSmem = kBytes + 1024;
};
static_assert(BandLayout::kDynSmem <= 232448, "band kernel shared memory");

// Position in the flattened tile list: tile i of sequence b, KV head kvh.
struct BandCursor {
  int32_t b, kvh, i;
  int32_t ntile;   // tiles of sequence b
  int32_t s0, L;   // first packed row and length of sequence b
  int32_t left;    // tiles of this CTA not yet passed (the current one included)
  int32_t run;     // 1 if this tile starts a run (first of the CTA or of its lane)
};

__device__ __forceinline__ void band_load_seq(BandCursor &c, const BandArgs &a) {
  c.s0 = __ldg(a.cu_seqlens + c.b);
  c.L = __ldg(a.cu_seqlens + c.b + 1) - c.s0;
  c.ntile = (c.L + kBandSeg - 1) / kBandSeg;
}

__device__ __forceinline__ void band_next(BandCursor &c, const BandArgs &a) {
  c.run = 0;
  if (--c.left <= 0) return;
  if (++c.i < c.ntile) return;
  c.i = 0;
  c.run = 1;
  if (++c.kvh < a.Hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
    band_load_seq(c, a);
  } while (c.ntile == 0 && c.b + 1 < a.batch);
}

// Window of the cursor's tile: nwin segments starting at segment i - nwin + 1.
__device__ __forceinline__ int32_t band_nwin(const BandCursor &c, const BandArgs &a) {
  return min(c.i + 1, a.nseg);
}

// Set-up (one warp): the exact number of tiles, this CTA's share of the
// flattened list and the (sequence, KV head, tile) it starts at.
__device__ void band_locate(const BandArgs &a, int32_t lane, int32_t *cur) {
  uint32_t ct = 0;
  for (int32_t b = lane; b < a.batch; b += 32) {
    const int32_t L = __ldg(a.cu_seqlens + b + 1) - __ldg(a.cu_seqlens + b);
    ct += static_cast<uint32_t>((L + kBandSeg - 1) / kBandSeg);
  }
  ct = __reduce_add_sync(0xffffffffu, ct);
  const int64_t T = int64_t(ct) * a.Hkv;
  const int64_t f0 = T * blockIdx.x / gridDim.x;
  const int64_t f1 = T * (blockIdx.x + 1) / gridDim.x;
  int32_t sb = 0, skvh = 0, si = 0;
  bool found = false;
  int64_t run = 0;
  for (int32_t base = 0; base < a.batch && !found && f1 > f0; base += 32) {
    const int32_t b = base + lane;
    int32_t c = 0;
    if (b < a.batch) {
      const int32_t L = __ldg(a.cu_seqlens + b + 1) - __ldg(a.cu_seqlens + b);
      c = (L + kBandSeg - 1) / kBandSeg;
    }
    const int64_t w = int64_t(c) * a.Hkv;
    int64_t incl = w;
#pragma unroll
    for (int32_t o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, w > 0 && run + incl > f0);
    if (m) {
      const int32_t j = __ffs(m) - 1;
      const int64_t incl_j = __shfl_sync(0xffffffffu, incl, j);
      const int64_t w_j = __shfl_sync(0xffffffffu, w, j);
      const int32_t c_j = __shfl_sync(0xffffffffu, c, j);
      const int64_t off = f0 - (run + incl_j - w_j);
      sb = base + j;
      skvh = static_cast<int32_t>(off / c_j);
      si = static_cast<int32_t>(off % c_j);
      found = true;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    cur[0] = sb;
    cur[1] = skvh;
    cur[2] = si;
    cur[3] = found ? static_cast<int32_t>(f1 - f0) : 0;
  }
}


// Mask of the N band columns k0 .. k0+N-1 of this thread's half held in r,
// by groups of 8: columns that are not visible (k - lo > span as unsigned)
// become -inf, unless the whole warp sees all 8 of the group.
template <int N>
__device__ __forceinline__ void band_mask(uint32_t (&r)[N], int32_t k0, int32_t lo, uint32_t span) {
  constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
  for (int32_t g = 0; g < N; g += 8) {
    const bool whole = static_cast<uint32_t>(k0 + g - lo) <= span &&
                       static_cast<uint32_t>(k0 + g + 7 - lo) <= span;
    if (!__all_sync(0xffffffffu, whole)) {
#pragma unroll
      for (int32_t k = 0; k < 8; ++k)
        if (static_cast<uint32_t>(k0 + g + k - lo) > span) r[g + k] = kNegInf;
    }
  }
}

// TMEM load of N (8 or 16) columns.
template <int N>
__device__ __forceinline__ void band_ld(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 16) tmem_ld16p(taddr, r);
  else tmem_ld8p(taddr, r);
  tmem_wait_ld();
  reg_fence<N>(r);
}

// Pass 1 on N columns at k0: mask, then the running maximum.
template <int N>
__device__ __forceinline__ void band_p1(uint32_t s_h, int32_t k0, int32_t lo, uint32_t span,
                                        float &mxa, float &mxb) {
  uint32_t r[N];
  band_ld<N>(s_h + k0, r);
  band_mask<N>(r, k0, lo, span);
#pragma unroll
  for (int32_t k = 0; k < N; k += 4) {
    mxa = fmax3(mxa, __uint_as_float(r[k]), __uint_as_float(r[k + 1]));
    mxb = fmax3(mxb, __uint_as_float(r[k + 2]), __uint_as_float(r[k + 3]));
  }
}

// Pass 2 on N columns at k0: P = 2^(s * scale * log2e - m) summed and stored
// as bf16 pairs at p_h + k0/2.
template <int N>
__device__ __forceinline__ void band_p2(uint32_t s_h, uint32_t p_h, int32_t k0, int32_t lo,
                                        uint32_t span, float2 sc2, float2 mneg2, float2 &sum2) {
  uint32_t r[N];
  band_ld<N>(s_h + k0, r);
  band_mask<N>(r, k0, lo, span);
#pragma unroll
  for (int32_t k = 0; k < N; k += 2) {
    const float2 y = ffma2(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), sc2, mneg2);
    const float2 pp = make_float2(ex2(y.x), ex2(y.y));
    sum2 = fadd2(sum2, pp);
    r[k >> 1] = pack_bf16x2(pp.x, pp.y);
  }
  if constexpr (N == 16) tmem_st8p(p_h + (k0 >> 1), r);
  else tmem_st4p(p_h + (k0 >> 1), r);
}

// Softmax + epilogue of one half of every row (half 0: band columns 0..71 and
// output dims 0..63; half 1: band columns 72..143 and output dims 64..127).
// Each of the two passes walks the 72 logits of the half in one chunk of 8 and
// four of 16, masking them in registers: pass 1 takes the maximum, pass 2
// forms P.  The two threads of a row swap their partial maximum of tile i and their partial sum of tile i-1
// through shared memory, paired by an mbarrier.  Both halves run the same code
// (half is a runtime value) to keep the hot loop small in the instruction cache.
__device__ __forceinline__ void band_softmax(const BandArgs &args, const BandCursor &c0,
                                             uint32_t tmem, uint32_t sbase, uint8_t *smem,
                                             volatile uint32_t *abort_flag) {
  using Ly = BandLayout;
  constexpr int32_t R = kBandRing;
  const uint32_t bars = sbase + Ly::kBarOff;
  auto B_SFULL = [&](uint32_t b) { return bars + (6 + 3 * R + b) * 8; };
  auto B_PFULL = [&](uint32_t b) { return bars + (6 + 3 * R + 2 + b) * 8; };
  const uint32_t B_PVDONE = bars + (6 + 3 * R + 4) * 8;
  const uint32_t B_OEMPTY = bars + (6 + 3 * R + 5) * 8;
  const int32_t warp = threadIdx.x >> 5;
  const int32_t half = warp >= 8 ? 1 : 0;
  const int32_t c0col = half * kBandHalf;  // first band column of this half
  const int32_t row = (warp & 3) * 32 + (threadIdx.x & 31);  // query row == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  auto B_PAIR = [&](uint32_t par) { return bars + (Ly::kPairBar + par * 4 + (warp & 3)) * 8; };
  float2 *xchg = reinterpret_cast<float2 *>(smem + Ly::kXchgOff);  // [parity][half][row]
  const int32_t t = row / kBandG, g = row % kBandG;
  const float sc = args.scale_log2;
  const int32_t W = args.window;
  const uint32_t o_t = tmem + lane_off + kTmemO + half * 64;
  uint32_t gt = 0;
  bool ok = true;
  // the tile whose epilogue is pending
  bool p_valid = false;
  size_t p_orow = 0;
  float p_m = 0.f, p_sk = 0.f, p_sum = 0.f;
  // sink of this thread's head, reloaded only when the KV head changes (a
  // global load in the loop would queue behind the epilogue's output stores)
  int32_t sk_kvh = -1;
  float sk_cur = 0.f;

  // Swap (partial max of this tile, partial sum of the previous tile) with the
  // other thread of the row; returns the other's pair.
  auto swap = [&](uint32_t tt, float mx, float sum, float2 &other) -> bool {
    const uint32_t par = tt & 1;
    xchg[(par * 2 + half) * 128 + row] = make_float2(mx, sum);
    tc_fence_before();
    mbar_arrive(B_PAIR(par));
    if (!wait_bar_warp(B_PAIR(par), (tt >> 1) & 1, abort_flag, 12)) return false;
    tc_fence_after();
    other = xchg[(par * 2 + (1 - half)) * 128 + row];
    return true;
  };

  // One pass per tile, plus a last pass that only finishes the last epilogue.
  BandCursor c = c0;
  for (uint32_t step = 0; ok; ++step) {
    const bool have = c.left > 0;  // a tile to run the softmax of
    if (!have && step == 0) break;
    float mx = -INFINITY, m = 0.f, sk2 = 0.f, sum = 0.f;
    bool rvalid = false;
    size_t orow = 0;
    uint32_t s_t = 0, buf = 0;
    int32_t lo = 0;
    uint32_t span = 0;  // visible band columns of this half: k - lo <= span (unsigned)
    if (have) {
      const int32_t head = c.kvh * kBandG + g;
      const int32_t pos = c.i * kBandSeg + t;
      rvalid = pos < c.L;
      orow = static_cast<size_t>(c.s0 + pos) * args.Hq + head;
      const int32_t nwin = band_nwin(c, args);
      const int32_t kstart = (c.i - nwin + 1) * kBandSeg;
      // visible band columns [lo, hi] (hi < nwin * 16: columns past the
      // window hold stale values and are masked), shifted to this half
      lo = max(0, pos - W + 1) - kstart - c0col;
      const int32_t hi = pos - kstart - c0col;
      span = static_cast<uint32_t>(hi - lo);
      if (!rvalid) { lo = 1 << 20; span = 0; }
      if (c.kvh != sk_kvh) {
        sk_kvh = c.kvh;
        sk_cur = __ldg(args.sink + head) * kLog2e;  // -inf stays -inf
      }
      sk2 = sk_cur;
      buf = gt & 1;
      if (!(ok = wait_bar_warp(B_SFULL(buf), (gt >> 1) & 1, abort_flag, 7))) break;
      tc_fence_after();
      s_t = tmem + lane_off + tmem_s_col(buf);
      // pass 1: the mask and the maximum, one TMEM load of 8 then four of 16
      // columns (compact loops: the kernel's speed is bound by its
      // instruction-cache footprint, and a TMEM load round trip costs only tens
      // of cycles); every load offset is a multiple of its size
      const uint32_t s_h = s_t + c0col;
      const int32_t k8 = half ? 0 : kBandHalf - 8;   // the 8-column chunk
      const int32_t k16 = half ? 8 : 0;              // the first 16-column chunk
      float mxa = -INFINITY, mxb = -INFINITY;
      band_p1<8>(s_h, k8, lo, span, mxa, mxb);
#pragma unroll 1
      for (int32_t i = 0; i < 4; ++i) band_p1<16>(s_h, k16 + 16 * i, lo, span, mxa, mxb);
      mx = fmaxf(mxa, mxb);
    }
    float2 other = make_float2(-INFINITY, 0.f);
    if (!(ok = swap(step, mx, p_sum, other))) break;
    if (have) {
      // eq. (2): m = max(max_j a_ij, sink), in the log2 domain (scale > 0)
      m = fmaxf(fmaxf(mx, other.x) * sc, sk2);
      const float mneg = m == -INFINITY ? 0.f : -m;
      // pass 2: P = 2^(s * scale * log2e - m) as bf16 pairs; P of band column
      // k lands at TMEM column kBandPCol + k/2, so each half's P covers only
      // its own S columns (half 0: 36..71, half 1: 72..107); walking the
      // chunks downwards (half 0: 64, 48, 32, 16, 0) or upwards (half 1: 0, 8,
      // 24, 40, 56) overwrites only columns that were already read
      const float2 sc2 = make_float2(sc, sc), mneg2 = make_float2(mneg, mneg);
      float2 sum2 = make_float2(0.f, 0.f);
      const uint32_t s_h = s_t + c0col;
      const uint32_t p_h = s_t + kBandPCol + static_cast<uint32_t>(c0col >> 1);
      const int32_t k8 = half ? 0 : kBandHalf - 8;
      band_p2<8>(s_h, p_h, k8, lo, span, sc2, mneg2, sum2);
#pragma unroll 1
      for (int32_t i = 0; i < 4; ++i) {
        const int32_t k0 = half ? 8 + 16 * i : 48 - 16 * i;
        band_p2<16>(s_h, p_h, k0, lo, span, sc2, mneg2, sum2);
      }
      sum = sum2.x + sum2.y;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(B_PFULL(buf));
    }
    if (step > 0) {
      // ---------------- epilogue of the previous tile (eqs. (2)-(3)):
      // o = O / l with l = 2^(sink - m) + sum_j P_j, lse = (m + log2 l) ln 2
      if (!(ok = wait_bar_warp(B_PVDONE, (step - 1) & 1, abort_flag, 9))) break;
      tc_fence_after();
      const float l = (p_sk == -INFINITY ? 0.f : ex2(p_sk - p_m)) + (p_sum + other.y);
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      uint32_t w[32];  // this half-row as bf16 pairs: four 32-byte sectors of 8 words
      {
        uint32_t o[64];
        tmem_ld32p(o_t, o);
        tmem_ld32p(o_t + 32, o + 32);
        tmem_wait_ld();
        reg_fence<64>(o);
        // O is in registers: the next PV may overwrite it
        tc_fence_before();
        mbar_arrive(B_OEMPTY);
#pragma unroll
        for (int32_t e = 0; e < 32; ++e) {
          const float2 v = fmul2(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])),
                                 make_float2(inv_l, inv_l));
          w[e] = pack_bf16x2(v.x, v.y);
        }
      }
      // Each half-row is one 128-byte line of out, stored as its four 32-byte
      // sectors.  (Exchanging sectors within lane quads so that each store
      // writes whole lines cost the softmax warps more time than it saved.)
      if (p_valid && SA_OUT(p_orow, args.n_rows, 0x11)) {
        __nv_bfloat16 *line = args.out + p_orow * kDv + half * 64;
#pragma unroll
        for (int32_t pq = 0; pq < 4; ++pq) {
          uint32_t (&sec)[8] = *reinterpret_cast<uint32_t(*)[8]>(w + 8 * pq);
          if (args.out_v8) {
            st_global_v8(line + pq * 16, sec);
          } else {
            uint4 *d4 = reinterpret_cast<uint4 *>(line + pq * 16);
            d4[0] = make_uint4(sec[0], sec[1], sec[2], sec[3]);
            d4[1] = make_uint4(sec[4], sec[5], sec[6], sec[7]);
          }
        }
      }
      if (p_valid && half == 0 && SA_OUT(p_orow, args.n_rows, 0x12))
        args.lse[p_orow] = l > 0.f ? (p_m + __log2f(l)) * kLn2 : -INFINITY;
    }
    if (!have) break;
    p_valid = rvalid;
    p_orow = orow;
    p_m = m;
    p_sk = sk2;
    p_sum = sum;
    ++gt;
    band_next(c, args);
  }
}

__global__ void __launch_bounds__(kBandThreads, 1)
    sinkattn_band_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ BandArgs args) {
  using Ly = BandLayout;
  constexpr int32_t R = kBandRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int32_t warp = threadIdx.x >> 5;
  const int32_t lane = threadIdx.x & 31;

  auto bar = [&](uint32_t i) { return sbase + Ly::kBarOff + i * 8; };
  auto B_QFULL = [&](uint32_t s) { return bar(s); };
  auto B_QREADY = [&](uint32_t s) { return bar(2 + s); };
  auto B_QEMPTY = [&](uint32_t s) { return bar(4 + s); };
  auto B_SEGFULL = [&](uint32_t s) { return bar(6 + s); };
  auto B_SEGREADY = [&](uint32_t s) { return bar(6 + R + s); };
  auto B_SEGEMPTY = [&](uint32_t s) { return bar(6 + 2 * R + s); };
  auto B_SFULL = [&](uint32_t b) { return bar(6 + 3 * R + b); };
  auto B_PFULL = [&](uint32_t b) { return bar(6 + 3 * R + 2 + b); };
  const uint32_t B_PVDONE = bar(6 + 3 * R + 4);
  const uint32_t B_OEMPTY = bar(6 + 3 * R + 5);
  const uint32_t B_DRAIN = bar(6 + 3 * R + 6);

  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Ly::kMiscOff + 4);
  int32_t *cur_smem = reinterpret_cast<int32_t *>(smem + Ly::kMiscOff + 16);
  unsigned long long *turns = reinterpret_cast<unsigned long long *>(smem + Ly::kTurnsOff);

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < 2; ++s) {
      mbar_init(B_QFULL(s), 1);
      mbar_init(B_QREADY(s), 128);
      mbar_init(B_QEMPTY(s), 1);
      mbar_init(B_SFULL(s), 1);
      mbar_init(B_PFULL(s), 256);
    }
    for (uint32_t s = 0; s < R; ++s) {
      mbar_init(B_SEGFULL(s), 1);
      mbar_init(B_SEGREADY(s), 128);
      mbar_init(B_SEGEMPTY(s), 1);
    }
    mbar_init(B_PVDONE, 1);
    mbar_init(B_OEMPTY, 256);
    mbar_init(B_DRAIN, 1);
    for (uint32_t i = 0; i < 8; ++i) mbar_init(bar(Ly::kPairBar + i), 64);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) turns[threadIdx.x] = args.rope_turns[threadIdx.x];
  if (warp == 2) {
    tmem_alloc(sbase + Ly::kMiscOff, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 3) band_locate(args, lane, cur_smem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  BandCursor c0;
  c0.b = cur_smem[0];
  c0.kvh = cur_smem[1];
  c0.i = cur_smem[2];
  c0.left = cur_smem[3];
  c0.run = 1;
  if (c0.left > 0) band_load_seq(c0, args);
  if (warp < 4) {
    if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0 && c0.left > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t gq = 0, gseg = 0;
      bool ok = true;
      for (BandCursor c = c0; ok && c.left > 0; band_next(c, args)) {
        const uint32_t qs = gq & 1;
        if (!(ok = wait_bar(B_QEMPTY(qs), ((gq >> 1) & 1) ^ 1, abort_flag, 1))) break;
        mbar_arrive_expect_tx(B_QFULL(qs), 3u * kQBoxBytes);
        const uint32_t qdst = sbase + Ly::kQOff + qs * kQStageBytes;
        const int32_t qrow = c.s0 + c.i * kBandSeg;
#pragma unroll
        for (int cc = 0; cc < 3; ++cc)
          tma_load_3d(qdst + cc * kQBoxBytes, &tm_q, cc * 64, c.kvh * kBandG, qrow, B_QFULL(qs));
        ++gq;
        const int32_t nwin = band_nwin(c, args);
        const int32_t nload = c.run ? nwin : 1;
        for (int32_t j = 0; j < nload; ++j) {
          const int32_t seg = c.i - nload + 1 + j;
          const uint32_t slot = gseg % R;
          if (!(ok = wait_bar(B_SEGEMPTY(slot), ((gseg / R) & 1) ^ 1, abort_flag, 2))) break;
          mbar_arrive_expect_tx(B_SEGFULL(slot), 5u * Ly::kSegBox);
          const int32_t krow = c.s0 + seg * kBandSeg;
#pragma unroll
          for (int cc = 0; cc < 3; ++cc)
            tma_load_3d(sbase + Ly::kKOff + cc * Ly::kRingBox + slot * Ly::kSegBox, &tm_k, cc * 64,
                        c.kvh, krow, B_SEGFULL(slot));
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            tma_load_3d(sbase + Ly::kVOff + cc * Ly::kRingBox + slot * Ly::kSegBox, &tm_v, cc * 64,
                        c.kvh, krow, B_SEGFULL(slot));
          ++gseg;
        }
      }
      // Drain: the last copy into each stage and slot must land before the CTA exits.
      for (uint32_t s = 0; s < 2; ++s)
        if (gq > s) drain_wait(B_QFULL(s), ((gq - 1 - s) >> 1) & 1);
      for (uint32_t s = 0; s < R; ++s)
        if (gseg > s) drain_wait(B_SEGFULL(s), ((gseg - 1 - s) / R) & 1);
    }
    } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0 && c0.left > 0) {
      constexpr uint32_t kIdescPV = idesc_f32acc(128, kDv, 1, 0, 1);
      // Shared-memory matrix descriptors (128-byte swizzle, SBO = 1024 B), as
      // (low, high) words: the low word holds start address >> 4 and LBO >> 4,
      // so every operand offset below is a single 32-bit add.
      constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
      const uint32_t q_lo = ((sbase + Ly::kQOff) >> 4) | (1u << 16);
      const uint32_t k_lo = ((sbase + Ly::kKOff) >> 4) | (1u << 16);
      // V is MN-major: LBO = one ring box (the two 64-column halves of dv)
      const uint32_t v_lo = ((sbase + Ly::kVOff) >> 4) | ((Ly::kRingBox >> 4) << 16);
      constexpr uint32_t kSegLo = Ly::kSegBox >> 4;
      const uint32_t rot = args.rope_on ? 0u : 1u;  // rotated dims are fp16
      uint32_t gt = 0, gseg = 0;
      bool ok = true;
#ifdef SINKATTN_TEST_HOOKS
      // B_DRAIN completes only after a commit issued when every MMA is out,
      // which has not happened yet: this wait can only run out
      if (g_test_stall_ns) ok = wait_bar_slow(B_DRAIN, 0, abort_flag, 0x7E, g_test_stall_ns);
#endif
      // the previous tile, whose PV is issued after the next tile's QK^T
      int32_t p_nwin = 0;
      uint32_t p_slot = 0;
      auto issue_pv = [&](uint32_t t, int32_t nwin, uint32_t slot, int32_t nfree) -> bool {
        const uint32_t buf = t & 1;
        if (!wait_bar(B_PFULL(buf), (t >> 1) & 1, abort_flag, 4)) return false;
        tc_fence_after();
        if (!wait_bar(B_OEMPTY, (t & 1) ^ 1, abort_flag, 5)) return false;
        tc_fence_after();
        const uint32_t p_t = tmem + tmem_s_col(buf) + kBandPCol;
        uint32_t sl = slot;
        for (int32_t kk = 0; kk < nwin; ++kk) {
          mma_ts2(tmem + kTmemO, p_t + kk * 8, v_lo + sl * kSegLo, kDescHi, kIdescPV,
                  kk > 0 ? 1u : 0u);
          sl = sl + 1 == R ? 0 : sl + 1;
        }
        sl = slot;
        for (int32_t kk = 0; kk < nfree; ++kk) {
          mma_commit(B_SEGEMPTY(sl));
          sl = sl + 1 == R ? 0 : sl + 1;
        }
        mma_commit(B_PVDONE);
        return true;
      };
      for (BandCursor c = c0; ok && c.left > 0; band_next(c, args)) {
        const int32_t nwin = band_nwin(c, args);
        const int32_t nload = c.run ? nwin : 1;
        if (gt > 0 && c.run) {
          // a new run reloads the whole band: the previous tile's segments must
          // be released (its PV issued) before this tile's loads can land
          if (!(ok = issue_pv(gt - 1, p_nwin, p_slot, p_nwin))) break;
        }
        const uint32_t qs = gt & 1;
        if (!(ok = wait_bar(B_QREADY(qs), (gt >> 1) & 1, abort_flag, 3))) break;
        for (int32_t j = 0; j < nload && ok; ++j) {
          const uint32_t g = gseg + j;
          ok = wait_bar(B_SEGREADY(g % R), (g / R) & 1, abort_flag, 6);
        }
        if (!ok) break;
        tc_fence_after();
        gseg += nload;
        const uint32_t slot0 = (gseg - nwin) % R;
        const uint32_t buf = gt & 1;
        const int32_t n1 = min(nwin, R - static_cast<int32_t>(slot0));
        const int32_t n2 = nwin - n1;
        const uint32_t id1 = idesc_f32acc(128, n1 * kBandSeg, 1, 0, 0);
        const uint32_t id1r = idesc_f32acc(128, n1 * kBandSeg, rot, 0, 0);
        const uint32_t id2 = idesc_f32acc(128, (n2 > 0 ? n2 : 1) * kBandSeg, 1, 0, 0);
        const uint32_t id2r = idesc_f32acc(128, (n2 > 0 ? n2 : 1) * kBandSeg, rot, 0, 0);
        const uint32_t a_lo = q_lo + qs * (kQStageBytes >> 4);
        const uint32_t b1_lo = k_lo + slot0 * kSegLo;
        const uint32_t s_t = tmem + tmem_s_col(buf);
        // S = Q K^T: 12 k-steps of 16 dims (3 boxes of 64); when the band wraps
        // the end of the ring, segments slot0.. and 0.. are two MMAs
#pragma unroll
        for (int kstep = 0; kstep < kDqk / 16; ++kstep) {
          const uint32_t box = kstep >> 2, off = (kstep & 3) * 32;
          const uint32_t ao = (box * kQBoxBytes + off) >> 4;
          const uint32_t bo = (box * Ly::kRingBox + off) >> 4;
          mma_ss2(s_t, a_lo + ao, kDescHi, b1_lo + bo, kDescHi, box == 0 ? id1r : id1,
                  kstep > 0 ? 1u : 0u);
          if (n2 > 0)
            mma_ss2(s_t + n1 * kBandSeg, a_lo + ao, kDescHi, k_lo + bo, kDescHi,
                    box == 0 ? id2r : id2, kstep > 0 ? 1u : 0u);
        }
        mma_commit(B_SFULL(buf));
        mma_commit(B_QEMPTY(qs));
        if (gt > 0 && !c.run) {
          // same lane: the oldest segment of the previous band leaves the window
          // once the band is full
          const int32_t nfree = nwin == p_nwin ? 1 : 0;
          if (!(ok = issue_pv(gt - 1, p_nwin, p_slot, nfree))) break;
        }
        p_nwin = nwin;
        p_slot = slot0;
        ++gt;
      }
      if (ok && gt > 0) ok = issue_pv(gt - 1, p_nwin, p_slot, p_nwin);
      if (gt > 0) {
        mma_commit(B_DRAIN);
        drain_wait(B_DRAIN, 0);
      }
    }
    }
  } else if (warp < 12) {
    // ============================================================ softmax + epilogue
    // Tile i's softmax runs before tile i-1's epilogue, so these warps never
    // wait on a PV: by the time tile i's P is stored, PV(i-1) has long finished.
    band_softmax(args, c0, tmem, sbase, smem, abort_flag);
  } else {
    // ============================================================ RoPE
    const int32_t tid = threadIdx.x - 384;
    uint32_t gq = 0, gseg = 0;
    bool ok = true;
    for (BandCursor c = c0; ok && c.left > 0; band_next(c, args)) {
      const uint32_t qs = gq & 1;
      if (!(ok = wait_bar_warp(B_QFULL(qs), (gq >> 1) & 1, abort_flag, 10))) break;
      if (args.rope_on)
        band_rope_q(smem + Ly::kQOff + qs * kQStageBytes, min(kBandSeg, c.L - c.i * kBandSeg),
                    c.i * kBandSeg, args.rope_style, turns, tid);
      fence_proxy_async_smem();
      mbar_arrive(B_QREADY(qs));
      ++gq;
      const int32_t nwin = band_nwin(c, args);
      const int32_t nload = c.run ? nwin : 1;
      for (int32_t j = 0; j < nload; ++j) {
        const int32_t seg = c.i - nload + 1 + j;
        const uint32_t slot = gseg % R;
        if (!(ok = wait_bar_warp(B_SEGFULL(slot), (gseg / R) & 1, abort_flag, 11))) break;
        if (args.rope_on)
          rope_k_rows(smem + Ly::kKOff + slot * Ly::kSegBox, kBandSeg, seg * kBandSeg,
                      args.rope_style, turns, tid);
        fence_proxy_async_smem();
        mbar_arrive(B_SEGREADY(slot));
        ++gseg;
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
