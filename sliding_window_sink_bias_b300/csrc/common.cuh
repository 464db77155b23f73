// common.cuh -- pieces shared by the attention kernels: constants, the device
// status word, bounded mbarrier waits, exact RoPE angles and the in-SMEM
// rotation of 128B-swizzled rows.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "ptx.cuh"

namespace sa {

constexpr int kThreads = 384;
constexpr int kDqk = 192;
constexpr int kDv = 128;
constexpr uint32_t kRowBytes = 128;                     // one 64-element bf16 row of a box
constexpr uint32_t kQBoxBytes = 128 * kRowBytes;        // 128 packed query rows
constexpr uint32_t kQStageBytes = 3 * kQBoxBytes;       // dims 0..191
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t tmem_s_col(uint32_t buf) { return buf ? 192u : 0u; }
constexpr uint32_t kTmemO = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitLimitNs = 4000000000ull;        // 4 s per wait
constexpr uint64_t kDrainLimitNs = 200000000ull;        // 0.2 s to drain after an abort

// Bounded mbarrier wait, slow path: the timed loop.  Returns false if this CTA
// is aborting (another wait gave up) or this wait runs past limit_ns, which
// then records SINKATTN_ETIMEOUT and the site in the status word and sets the
// CTA's abort flag.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity,
                                           volatile uint32_t *abort_flag, uint32_t site,
                                           uint64_t limit_ns = kWaitLimitNs) {
  // each try_wait sleeps up to its suspend hint (1 ms), so checking the clock
  // and the abort flag once per round costs nothing
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1u;
      status_record(1u, site, 8);
      return false;
    }
  }
}

// Bounded mbarrier wait.  A phase that has already completed is seen by the
// non-blocking test; otherwise the first try_wait (which itself sleeps up to
// its hint) almost always succeeds.  The timed loop lives out of line so the
// hot loops stay small in the instruction cache.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                         uint32_t site) {
  if (mbar_test_wait(bar, parity)) return true;
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, abort_flag, site);
}
// Warp-uniform form: every lane polls, then the warp agrees, so warp-collective
// tcgen05.ld/st that follow never run with part of the warp gone.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              volatile uint32_t *abort_flag, uint32_t site) {
  const bool ok = wait_bar(bar, parity, abort_flag, site);
  return __all_sync(0xffffffffu, ok);
}

#ifdef SINKATTN_TEST_HOOKS
// Test builds only (never in the product library): when the host sets it, the
// MMA thread of the next band-kernel launches first waits, for at most this
// many nanoseconds, on a barrier that nothing can complete yet, so that the
// timeout, abort and drain path runs without any fault.
__device__ uint64_t g_test_stall_ns;
#endif

// Wait used only while draining: ignores the abort flag, short limit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainLimitNs) {
      status_record(1u, 0xFFu, 8);
      return;
    }
  }
}

// cos/sin of pos * theta_t from a 64-bit fixed-point angle in turns: the product
// wraps modulo one full turn exactly, so the angle is exact before the final
// conversion to a float in [-pi, pi).
__device__ __forceinline__ void rope_cs(int32_t pos, unsigned long long turns_fp, float &c,
                                        float &s) {
  const unsigned long long prod =
      static_cast<unsigned long long>(static_cast<long long>(pos)) * turns_fp;
  const int32_t hi = static_cast<int32_t>(prod >> 32);
  const float ang = static_cast<float>(hi) * 1.4629180792671596e-09f;  // 2 pi / 2^32
  __sincosf(ang, &s, &c);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The rotated dims 0..63 are written back as fp16, not bf16: the 64-dim part of
// q.k then runs as its own fp16 x fp16 MMA k-steps (fp32 accumulate), and the
// rotation's re-rounding error drops 8-fold (11 vs 8 significant bits).  The
// one exception is a query tile multiplied with keys a cache already holds
// rotated in bf16 (the two operands of one MMA share a type): kBf16 = true.
template <bool kBf16>
__device__ __forceinline__ uint32_t pack_rot(float lo, float hi) {
  if constexpr (kBf16) return pack_bf16x2(lo, hi);
  else return pack_f16x2(lo, hi);
}

// Rotate the four (2t, 2t+1) pairs stored in one 16-byte chunk (pairs 4c..4c+3).
template <bool kBf16 = false>
__device__ __forceinline__ void rot_chunk_interleaved(uint4 *p, const float (&cs)[4],
                                                      const float (&sn)[4]) {
  uint4 v = *p;
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x = bf16lo(w[e]), y = bf16hi(w[e]);
    w[e] = pack_rot<kBf16>(x * cs[e] - y * sn[e], x * sn[e] + y * cs[e]);
  }
  *p = make_uint4(w[0], w[1], w[2], w[3]);
}

// Rotate the eight (t, t+32) pairs held by chunk c (dims 8c..8c+7) and chunk
// c+4 (dims 32+8c..32+8c+7).
template <bool kBf16 = false>
__device__ __forceinline__ void rot_chunks_half(uint4 *pa, uint4 *pb, const float (&cs)[8],
                                                const float (&sn)[8]) {
  uint4 va = *pa, vb = *pb;
  uint32_t a[4] = {va.x, va.y, va.z, va.w};
  uint32_t b[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x0 = bf16lo(a[e]), y0 = bf16lo(b[e]);
    const float x1 = bf16hi(a[e]), y1 = bf16hi(b[e]);
    const float c0 = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
    a[e] = pack_rot<kBf16>(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
    b[e] = pack_rot<kBf16>(x0 * s0 + y0 * c0, x1 * s1 + y1 * c1);
  }
  *pa = make_uint4(a[0], a[1], a[2], a[3]);
  *pb = make_uint4(b[0], b[1], b[2], b[3]);
}

// Address of 16-byte chunk c of row r in a 128B-swizzled box (1024-byte aligned).
__device__ __forceinline__ uint4 *swz_chunk(uint8_t *box, int32_t r, int32_t c) {
  return reinterpret_cast<uint4 *>(box + r * kRowBytes + ((c ^ (r & 7)) << 4));
}

// RoPE on dims 0..63 (box 0) of a Q tile of packed rows r = t * G + g: the
// n_tok tokens at positions pos0 + t share their angles, so each (token, chunk)
// unit computes its angles once and rotates all G heads.  nthr threads (128
// unless given).  kBf16: store the rotated dims as bf16 instead of fp16.
template <bool kBf16 = false>
__device__ void rope_q_tile(uint8_t *box0, int32_t G, int32_t n_tok, int32_t pos0,
                            int32_t rope_style, const unsigned long long *turns, int32_t tid,
                            int32_t nthr = 128) {
  if (n_tok <= 0) return;
  const int32_t nch = rope_style == 0 ? 8 : 4;
  const int32_t units = n_tok * nch;
  const int32_t hsplit = units >= nthr ? 1 : min(G, nthr / units);
  const int32_t hper = (G + hsplit - 1) / hsplit;
  for (int32_t u = tid; u < units * hsplit; u += nthr) {
    const int32_t hs = u / units, tc = u % units;
    const int32_t t = tc / nch, c = tc % nch;
    const int32_t pos = pos0 + t;
    const int32_t g0 = hs * hper, g1 = min(G, g0 + hper);
    if (rope_style == 0) {
      float cs[4], sn[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) rope_cs(pos, turns[4 * c + e], cs[e], sn[e]);
      for (int32_t g = g0; g < g1; ++g)
        rot_chunk_interleaved<kBf16>(swz_chunk(box0, t * G + g, c), cs, sn);
    } else {
      float cs[8], sn[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) rope_cs(pos, turns[8 * c + e], cs[e], sn[e]);
      for (int32_t g = g0; g < g1; ++g) {
        const int32_t r = t * G + g;
        rot_chunks_half<kBf16>(swz_chunk(box0, r, c), swz_chunk(box0, r, c + 4), cs, sn);
      }
    }
  }
}

// RoPE on dims 0..63 (box 0) of `rows` keys at positions kpos0 + row.  128 threads.
__device__ void rope_k_rows(uint8_t *box0, int32_t rows, int32_t kpos0, int32_t rope_style,
                            const unsigned long long *turns, int32_t tid) {
  if (rope_style == 0) {
    for (int32_t u = tid; u < rows * 8; u += 128) {
      const int32_t r = u >> 3, c = u & 7;
      float cs[4], sn[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) rope_cs(kpos0 + r, turns[4 * c + e], cs[e], sn[e]);
      rot_chunk_interleaved(swz_chunk(box0, r, c), cs, sn);
    }
  } else {
    for (int32_t u = tid; u < rows * 4; u += 128) {
      const int32_t r = u >> 2, c = u & 3;
      float cs[8], sn[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) rope_cs(kpos0 + r, turns[8 * c + e], cs[e], sn[e]);
      rot_chunks_half(swz_chunk(box0, r, c), swz_chunk(box0, r, c + 4), cs, sn);
    }
  }
}

}  // namespace sa
