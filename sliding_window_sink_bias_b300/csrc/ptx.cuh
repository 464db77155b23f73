// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, TMA tensor loads,
// tcgen05 (5th-generation tensor core) MMA, TMEM allocation and TMEM <-> register
// moves.  Every wrapper maps to one PTX instruction; nothing here computes.
#pragma once
#include <cstdint>

namespace sa {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Device status word: bit 0 = a wait timed out, bits 8..15 = the wait site;
// bit 1 = a bounds check failed (checking builds only), bits 16..23 = its site.
// The first event of each kind names its site (later ones only see the bit set).
__device__ uint32_t g_status_word;
__device__ __noinline__ void status_record(uint32_t bit, uint32_t site, uint32_t shift) {
  if (!(atomicOr(&g_status_word, bit) & bit)) atomicOr(&g_status_word, (site & 0xFFu) << shift);
}

// ------------------------------------------------------------------ checks
// Checking builds (SINKATTN_CHECKS) test, before the access, every TMA copy's
// x coordinate and shared-memory destination, every tcgen05.ld/st and MMA
// operand's TMEM lane and columns, and every global store's index against its
// tensor's extent.  A failed check records its site and skips that one access:
// barrier arrivals and MMA commits still happen, so a failed check never
// leaves a wait unmet (a skipped TMA copy leaves its barrier short of bytes,
// and that wait ends at its time limit).  In other builds every check is the
// constant `true` and its operands are not even evaluated.
#ifdef SINKATTN_CHECKS
// Test hooks: output tensors seen as this many rows shorter, TMEM columns admitted.
__device__ int64_t g_check_row_shrink;
__device__ uint32_t g_check_tmem_cols = 512;
__device__ __noinline__ void check_failed(uint32_t site) { status_record(2u, site, 16); }
__device__ __forceinline__ bool sa_check(bool ok, uint32_t site) {
  if (!ok) check_failed(site);
  return ok;
}
// index i of a workspace tensor of n rows (or elements)
__device__ __forceinline__ bool sa_in(int64_t i, int64_t n, uint32_t site) {
  return sa_check(i >= 0 && i < n, site);
}
// index i of an output tensor (out, lse, gradients) of n rows
__device__ __forceinline__ bool sa_out(int64_t i, int64_t n, uint32_t site) {
  return sa_check(i >= 0 && i < n - g_check_row_shrink, site);
}
extern __shared__ uint8_t sa_check_dyn_smem[];  // aliases the kernel's dynamic shared memory
// [addr, addr + bytes) inside the CTA's dynamic shared memory
__device__ __forceinline__ bool smem_span_ok(uint32_t addr, uint32_t bytes) {
  uint32_t size;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
  const uint32_t lo = smem_addr(sa_check_dyn_smem);
  return addr >= lo && addr + bytes <= lo + size;
}
// a 32x32b tcgen05.ld/st of ncols columns: the warp's own lane quarter
__device__ __forceinline__ bool tmem_span_ok(uint32_t taddr, uint32_t ncols) {
  const uint32_t quarter = (threadIdx.x >> 5) & 3u;
  return (taddr >> 16) == 32u * quarter && (taddr & 0xFFFFu) + ncols <= g_check_tmem_cols;
}
#define SA_CHECK(cond, site) ::sa::sa_check((cond), (site))
#define SA_IN(i, n, site) ::sa::sa_in(static_cast<int64_t>(i), static_cast<int64_t>(n), (site))
#define SA_OUT(i, n, site) ::sa::sa_out(static_cast<int64_t>(i), static_cast<int64_t>(n), (site))
#else
#define SA_CHECK(cond, site) true
#define SA_IN(i, n, site) true
#define SA_OUT(i, n, site) true
#endif

// Check sites of the wrappers below (kernels use 0x10 and up).
constexpr uint32_t kSiteTmaCoord = 0x01, kSiteTmaDst = 0x02, kSiteTmemLd = 0x03,
                   kSiteTmemSt = 0x04, kSiteMmaD = 0x05, kSiteMmaA = 0x06, kSiteMmaB = 0x07,
                   kSiteMmaKind = 0x08;

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// Non-blocking test of the phase (no suspend).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Test the phase; if it is not complete the thread is suspended in hardware
// until it completes or the suspend-time hint (ns) runs out, so a waiting warp
// takes no issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------------------------ proxies
// Make generic-proxy writes to shared memory visible to the async proxy (TMA,
// tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int32_t c0, int32_t c1,
                                            int32_t c2, uint32_t bar) {
  // x must start on a 16-byte boundary (every map's x is a multiple of 64
  // elements here); the destination on a 128-byte boundary, in this CTA's buffer
  if (!SA_CHECK((c0 & 15) == 0, kSiteTmaCoord)) return;
  if (!SA_CHECK((dst & 127u) == 0 && smem_span_ok(dst, 128), kSiteTmaDst)) return;
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
#ifdef SINKATTN_CHECKS
// D: lane 0, N columns; A and B of one type (kind::f16 faults on a mix).
__device__ __forceinline__ bool mma_d_ok(uint32_t d_tmem, uint32_t idesc) {
  const uint32_t n = ((idesc >> 17) & 0x3Fu) << 3;
  return sa_check((d_tmem >> 16) == 0 && (d_tmem & 0xFFFFu) + n <= g_check_tmem_cols, kSiteMmaD) &&
         sa_check(((idesc >> 7) & 7u) == ((idesc >> 10) & 7u), kSiteMmaKind);
}
// a shared-memory operand: its start address (low 14 bits of the descriptor,
// in 16-byte units) inside this CTA's buffer
__device__ __forceinline__ bool mma_smem_ok(uint32_t desc_lo, uint32_t site) {
  return sa_check(smem_span_ok((desc_lo & 0x3FFFu) << 4, 32), site);
}
// A in TMEM: lane 0 and its K = 16 columns of 16-bit pairs (8 columns)
__device__ __forceinline__ bool mma_a_tmem_ok(uint32_t a_tmem) {
  return sa_check((a_tmem >> 16) == 0 && (a_tmem & 0xFFFFu) + 8 <= g_check_tmem_cols, kSiteMmaA);
}
#define SA_MMA_SS_OK(d, idesc, alo, blo) \
  (::sa::mma_d_ok((d), (idesc)) && ::sa::mma_smem_ok((alo), kSiteMmaA) && \
   ::sa::mma_smem_ok((blo), kSiteMmaB))
#define SA_MMA_TS_OK(d, idesc, a, blo) \
  (::sa::mma_d_ok((d), (idesc)) && ::sa::mma_a_tmem_ok(a) && ::sa::mma_smem_ok((blo), kSiteMmaB))
#else
#define SA_MMA_SS_OK(d, idesc, alo, blo) true
#define SA_MMA_TS_OK(d, idesc, a, blo) true
#endif

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  if (!SA_MMA_SS_OK(d_tmem, idesc, static_cast<uint32_t>(a_desc), static_cast<uint32_t>(b_desc)))
    return;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// As mma_ss, with each descriptor given as its low and high 32-bit words (the
// start-address field sits in the low word, so offsets are one 32-bit add).
__device__ __forceinline__ void mma_ss2(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                        uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  if (!SA_MMA_SS_OK(d_tmem, idesc, a_lo, b_lo)) return;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts2(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                        uint32_t idesc, uint32_t accumulate) {
  if (!SA_MMA_TS_OK(d_tmem, idesc, a_tmem, b_lo)) return;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  if (!SA_MMA_TS_OK(d_tmem, idesc, a_tmem, static_cast<uint32_t>(b_desc))) return;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 32), kSiteTmemLd)) {
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 32 bit, 16 consecutive columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[32]) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 16), kSiteTmemLd)) {
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 32), kSiteTmemSt)) return;
#endif
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 16), kSiteTmemSt)) return;
#endif
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[16]) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 8), kSiteTmemSt)) return;
#endif
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}


// Pointer forms of the TMEM moves (r must index a register array with constant
// offsets after unrolling).
__device__ __forceinline__ void tmem_ld32p(uint32_t taddr, uint32_t *r) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 32), kSiteTmemLd)) {
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16p(uint32_t taddr, uint32_t *r) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 16), kSiteTmemLd)) {
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32p(uint32_t taddr, const uint32_t *r) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 32), kSiteTmemSt)) return;
#endif
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st8p(uint32_t taddr, const uint32_t *r) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 8), kSiteTmemSt)) return;
#endif
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_ld8p(uint32_t taddr, uint32_t *r) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 8), kSiteTmemLd)) {
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld4p(uint32_t taddr, uint32_t *r) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 4), kSiteTmemLd)) {
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16p(uint32_t taddr, const uint32_t *r) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 16), kSiteTmemSt)) return;
#endif
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st4p(uint32_t taddr, const uint32_t *r) {
#ifdef SINKATTN_CHECKS
  if (!sa_check(tmem_span_ok(taddr, 4), kSiteTmemSt)) return;
#endif
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
      : "memory");
}

// Named barrier over `count` threads (whole warps).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Ties registers filled by tcgen05.ld to the tcgen05.wait::ld before it: an empty
// volatile asm that "rewrites" each register keeps the compiler from moving
// their uses above the wait.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t *r) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Move registers between warpgroups (every thread of the warpgroup executes it).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// One 32-byte global store (a whole sector); addr must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *addr, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(addr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// ------------------------------------------------------------------ math
// Packed fp32 pairs (two lanes of one 64-bit register): d = a * b + c, a + b, a * b.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> packed fp16x2 (round to nearest even); `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor for tcgen05.mma with the 128-byte swizzle:
// start address, leading- and stride-dimension byte offsets (all >> 4), the
// sm_100-family descriptor version (bit 46) and the layout type (2 = 128B swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, A and B both bf16
// (ab_bf16 = 1) or both fp16 (ab_bf16 = 0), the major-ness of A and B
// (0 = K-major, 1 = MN-major), N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t idesc_f32acc(uint32_t m, uint32_t n, uint32_t ab_bf16,
                                                    uint32_t a_mn_major, uint32_t b_mn_major) {
  return (1u << 4)             // D format: f32
         | (ab_bf16 << 7)      // A format: 1 = bf16, 0 = f16
         | (ab_bf16 << 10)     // B format: same as A
         | (a_mn_major << 15)  //
         | (b_mn_major << 16)  //
         | ((n >> 3) << 17)    //
         | ((m >> 4) << 24);
}

}  // namespace sa
