// sinkattn.cu -- host side of the C ABI declared in include/sinkattn.h:
// argument checks, TMA tensor maps, tile-schedule parameters and launches.
// All arithmetic of the attention runs in the kernels of attn_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "attn_kernel.cuh"
#include "band_kernel.cuh"
#include "decode_kernel.cuh"
#include "backward_kernel.cuh"
#include "causal_kernel.cuh"
#include "sinkattn.h"

namespace {

// Raise a kernel's dynamic shared-memory limit on the current device once: the
// attribute stays with the context, and setting it before every launch costs a
// driver call per launch.  A failed launch forgets the kernel, so the next call
// sets it again (a device reset clears it).
std::mutex g_smem_attr_mu;
std::vector<std::pair<const void *, uint64_t>> g_smem_attr_done;  // kernel, devices set (bit)

bool smem_attr_set(const void *kern, uint64_t bit) {
  std::lock_guard<std::mutex> lock(g_smem_attr_mu);
  for (auto &e : g_smem_attr_done)
    if (e.first == kern) return (e.second & bit) != 0;
  return false;
}

void smem_attr_mark(const void *kern, uint64_t bit, bool set) {
  std::lock_guard<std::mutex> lock(g_smem_attr_mu);
  for (auto &e : g_smem_attr_done)
    if (e.first == kern) {
      e.second = set ? (e.second | bit) : (e.second & ~bit);
      return;
    }
  if (set) g_smem_attr_done.emplace_back(kern, bit);
}

template <typename Kernel>
sinkattn_status smem_attr_once(Kernel kern, uint32_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SINKATTN_ECUDA;
  const void *key = reinterpret_cast<const void *>(kern);
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (bit != 0 && smem_attr_set(key, bit)) return SINKATTN_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return SINKATTN_ECUDA;
  if (bit != 0) smem_attr_mark(key, bit, true);
  return SINKATTN_OK;
}

// The status of a launch just made; on failure the kernel's attribute is set
// again at its next launch.
template <typename Kernel>
sinkattn_status launched(Kernel kern) {
  if (cudaGetLastError() == cudaSuccess) return SINKATTN_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev < 64)
    smem_attr_mark(reinterpret_cast<const void *>(kern), 1ull << dev, false);
  return SINKATTN_ECUDA;
}


using sa::AttnArgs;
using sa::Layout;

constexpr int32_t kVersion = 200;  // 0.2.0: sinkattn_params gained k_rotated
constexpr int32_t kBNWide = 144;   // one key block covers a 128-key window + 16-token tile
constexpr int32_t kBN = 128;
constexpr uint32_t kQBoxBytesHost = 128 * 128;  // one 64-dim box of a 128-row Q tile

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool pow2_upto_128(int32_t x) { return x >= 1 && x <= 128 && (x & (x - 1)) == 0; }

// ----------------------------------------------------------------- CUDA driver entry point
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A 3-D bf16 tensor map over rows of `heads` x `dim` elements: dims
// (dim, heads, rows) with a box of (64, box_heads, box_rows), 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t dim, uint64_t heads, uint64_t rows,
              uint32_t box_heads, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t gdim[3] = {dim, heads, rows};
  const cuuint64_t gstride[2] = {dim * 2, dim * heads * 2};
  const cuuint32_t box[3] = {64, box_heads, box_rows};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), gdim,
                        gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct DeviceInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

bool device_info(DeviceInfo &d) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  return true;
}

// RoPE angles as 64-bit fixed-point turns: theta_t = base^(-2t/64) (RoFormer
// frequencies over the 64 rotated dims, §2.1), stored as round(theta_t/(2 pi) * 2^64).
void fill_turns(AttnArgs &a, float rope_base) {
  for (int t = 0; t < 32; ++t) {
    const double theta = std::pow(static_cast<double>(rope_base), -2.0 * t / 64.0);
    const double turns = theta / (2.0 * M_PI);
    a.rope_turns[t] = static_cast<unsigned long long>(std::ldexp(turns, 64));
  }
}

sinkattn_status fill_common(AttnArgs &a, const sinkattn_params *p, float rope_base,
                            int32_t hq, int32_t hkv, int32_t window) {
  std::memset(&a, 0, sizeof a);
  a.Hq = hq;
  a.Hkv = hkv;
  a.G = hq / hkv;
  a.window = window;
  float scale = 1.0f / std::sqrt(192.0f);
  a.rope_on = 1;
  a.rope_style = 0;
  if (p) {
    if (p->scale != 0.f) scale = p->scale;
    a.rope_on = p->rope_off ? 0 : 1;
    a.rope_style = p->rope_style;
    if (p->rope_style != 0 && p->rope_style != 1) return SINKATTN_EINVAL;
    if (!(std::isfinite(scale))) return SINKATTN_EINVAL;
  }
  if (a.rope_on && !(rope_base > 0.f && std::isfinite(rope_base))) return SINKATTN_EINVAL;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  if (a.rope_on) fill_turns(a, rope_base);
  return SINKATTN_OK;
}

template <int BN, int NQ, int NKV>
sinkattn_status launch(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                       const AttnArgs &a, int grid, cudaStream_t stream) {
  using Ly = Layout<BN, NQ, NKV>;
  auto kern = sa::sinkattn_fwd_kernel<BN, NQ, NKV>;
  if (sinkattn_status st = smem_attr_once(kern, Ly::kDynSmem)) return st;
  kern<<<grid, sa::kThreads, Ly::kDynSmem, stream>>>(mq, mk, mv, a);
  return launched(kern);
}

// Sliding-window prefill with 8 query heads per KV head and W <= 128: the
// banded kernel with the K/V ring.
sinkattn_status launch_band(const void *q, const void *k, const void *v, const AttnArgs &a,
                            const int32_t *cu_seqlens, int32_t batch, int32_t total,
                            const DeviceInfo &dev, cudaStream_t stream) {
  sa::BandArgs b;
  std::memset(&b, 0, sizeof b);
  b.Hq = a.Hq;
  b.Hkv = a.Hkv;
  b.window = a.window;
  b.batch = batch;
  b.nseg = (a.window - 1 + sa::kBandSeg - 1) / sa::kBandSeg + 1;
  b.rope_on = a.rope_on;
  b.rope_style = a.rope_style;
  b.scale_log2 = a.scale_log2;
  b.out_v8 = aligned(a.out, 32) ? 1 : 0;
  b.cu_seqlens = cu_seqlens;
  b.sink = a.sink;
  b.out = a.out;
  b.lse = a.lse;
  b.n_rows = a.n_rows;
  std::memcpy(b.rope_turns, a.rope_turns, sizeof b.rope_turns);
  // upper bound of the tile count: sum_b ceil(L_b / 16) <= (total + 15 * batch) / 16
  const int64_t tiles = int64_t(a.Hkv) * ((int64_t(total) + 15 * int64_t(batch)) / sa::kBandSeg);
  if (tiles > INT32_MAX) return SINKATTN_EUNSUPPORTED;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, 192, a.Hq, total, sa::kBandG, sa::kBandSeg) ||
      !make_map(&mk, k, 192, a.Hkv, total, 1, sa::kBandSeg) ||
      !make_map(&mv, v, 128, a.Hkv, total, 1, sa::kBandSeg))
    return SINKATTN_ECUDA;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tiles, dev.sms)));
  auto kern = sa::sinkattn_band_kernel;
  if (sinkattn_status st = smem_attr_once(kern, sa::BandLayout::kDynSmem)) return st;
  kern<<<grid, sa::kBandThreads, sa::BandLayout::kDynSmem, stream>>>(mq, mk, mv, b);
  return launched(kern);
}

// Causal prefill, global or windowed, positive logit scale (except the band
// kernel's shapes): pairs of query tiles per CTA, longest first.
sinkattn_status launch_causal(const void *q, const void *k, const void *v, const AttnArgs &a,
                              const int32_t *cu_seqlens, int32_t batch, int32_t total,
                              int32_t max_seqlen, const DeviceInfo &dev, cudaStream_t stream) {
  sa::CausalArgs c;
  std::memset(&c, 0, sizeof c);
  c.Hq = a.Hq;
  c.Hkv = a.Hkv;
  c.G = a.G;
  c.window = a.window;
  c.T = 128 / a.G;
  c.batch = batch;
  c.max_seqlen = max_seqlen;
  c.npairs = (max_seqlen + 2 * c.T - 1) / (2 * c.T);
  const int64_t n_items = int64_t(batch) * a.Hkv * c.npairs;
  if (n_items > INT32_MAX) return SINKATTN_EUNSUPPORTED;
  c.n_items = static_cast<int32_t>(n_items);
  c.rope_on = a.rope_on;
  c.rope_style = a.rope_style;
  c.q_tx_bytes = 3u * kQBoxBytesHost;
  c.scale_log2 = a.scale_log2;
  c.out_v8 = aligned(a.out, 32) ? 1 : 0;
  c.cu_seqlens = cu_seqlens;
  c.sink = a.sink;
  c.out = a.out;
  c.lse = a.lse;
  c.n_rows = a.n_rows;
  std::memcpy(c.rope_turns, a.rope_turns, sizeof c.rope_turns);
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, 192, a.Hq, total, a.G, c.T) ||
      !make_map(&mk, k, 192, a.Hkv, total, 1, sa::kCauBN) ||
      !make_map(&mv, v, 128, a.Hkv, total, 1, sa::kCauBN))
    return SINKATTN_ECUDA;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(n_items, dev.sms)));
  auto kern = sa::sinkattn_causal_kernel;
  if (sinkattn_status st = smem_attr_once(kern, sa::CauLayout::kDynSmem)) return st;
  kern<<<grid, sa::kCauThreads, sa::CauLayout::kDynSmem, stream>>>(mq, mk, mv, c);
  return launched(kern);
}

struct DecodePlan {
  int32_t rows = 0;
  size_t tab_bytes = 0, bytes = 0;
};

// Decode workspace: one 64-bit ticket per unit (batch x KV heads, padded to
// 256 bytes), then 2 partial slots per CTA of R rows x (128 + 4) fp32, for at
// most sa::kDecMaxGrid CTAs.
DecodePlan decode_plan(int32_t batch, int32_t T, int32_t hq, int32_t hkv) {
  DecodePlan p;
  p.rows = T * (hq / hkv);
  p.tab_bytes = (static_cast<size_t>(batch) * hkv * sizeof(uint64_t) + 255) & ~size_t(255);
  p.bytes = p.tab_bytes +
            static_cast<size_t>(sa::kDecMaxGrid) * 2 * p.rows * (sa::kDv + 4) * sizeof(float);
  return p;
}

// A number for each decode call, different from every other call of this
// process (48 bits): the tickets of a call are told from the words earlier
// calls left in the workspace by it.  It starts at a value drawn from the
// clock and the address space, so another process that used the same memory
// is unlikely (2^-48 per ticket) to have left this call's number behind.
unsigned long long next_decode_epoch() {
  static std::atomic<unsigned long long> counter{
      (static_cast<unsigned long long>(
           std::chrono::steady_clock::now().time_since_epoch().count()) ^
       (reinterpret_cast<uintptr_t>(&counter) << 7)) & 0xFFFFFFFFFFFFull};
  unsigned long long e = counter.fetch_add(1) & 0xFFFFFFFFFFFFull;
  return e == 0 ? 1ull : e;
}

}  // namespace

extern "C" {

int32_t sinkattn_version(void) { return kVersion; }

// ----------------------------------------------------------------- backward
// Workspace: the rotated dims 0..63 of q and k, bf16 [total, Hq, 64] and
// [total, Hkv, 64],
// D fp32 [total, Hq], per-chunk sink-gradient partials fp32 [chunks, Hq];
// each region starts on 256 bytes.
struct BwdPlan {
  size_t q_rot = 0, k_rot = 0, D = 0, part = 0, bytes = 0;
  int32_t chunks = 0;
};

BwdPlan bwd_plan(int64_t total, int32_t hq, int32_t hkv) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  BwdPlan p;
  p.chunks = static_cast<int32_t>((total + sa::kBwdChunk - 1) / sa::kBwdChunk);
  p.q_rot = 0;
  p.k_rot = p.q_rot + up(static_cast<size_t>(total) * hq * 64 * 2);
  p.D = p.k_rot + up(static_cast<size_t>(total) * hkv * 64 * 2);
  p.part = p.D + up(static_cast<size_t>(total) * hq * 4);
  p.bytes = p.part + up(static_cast<size_t>(p.chunks > 0 ? p.chunks : 1) * hq * 4);
  return p;
}

size_t sinkattn_prefill_backward_workspace_size(int32_t total, int32_t num_q_heads,
                                                int32_t num_kv_heads) {
  if (total < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  return bwd_plan(total, num_q_heads, num_kv_heads).bytes;
}

sinkattn_status sinkattn_prefill_backward(const void *q, const void *k, const void *v,
                                          const float *sink, const int32_t *cu_seqlens,
                                          int32_t batch, int32_t total, int32_t max_seqlen,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t window, float rope_base,
                                          const sinkattn_params *params, const void *out,
                                          const float *lse, const void *dout, void *workspace,
                                          size_t workspace_bytes, void *dq, void *dk, void *dv,
                                          float *dsink, sinkattn_stream_t stream) {
  if (batch < 0 || total < 0 || max_seqlen < 0 || window < 0) return SINKATTN_EINVAL;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return SINKATTN_EINVAL;
  const int32_t G = num_q_heads / num_kv_heads;
  if (!pow2_upto_128(G) || G > 64) return SINKATTN_EUNSUPPORTED;
  if (num_q_heads > 65535 || num_kv_heads > 65535) return SINKATTN_EUNSUPPORTED;
  if (params && (params->kv_ring || params->k_rotated)) return SINKATTN_EINVAL;
  if (total > 0 && max_seqlen == 0) return SINKATTN_EINVAL;
  AttnArgs a;
  if (sinkattn_status st = fill_common(a, params, rope_base, num_q_heads, num_kv_heads, window))
    return st;
  if (!(a.scale_log2 > 0.f)) return SINKATTN_EINVAL;
  if (batch == 0 || total == 0) {
    if (!dsink) return SINKATTN_EINVAL;
    return cudaMemsetAsync(dsink, 0, sizeof(float) * num_q_heads,
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SINKATTN_OK
               : SINKATTN_ECUDA;
  }
  if (!q || !k || !v || !sink || !cu_seqlens || !out || !lse || !dout || !dq || !dk || !dv || !dsink)
    return SINKATTN_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(sink, 4) || !aligned(dsink, 4) || !aligned(cu_seqlens, 4))
    return SINKATTN_EINVAL;
  const BwdPlan plan = bwd_plan(total, num_q_heads, num_kv_heads);
  if (!workspace || workspace_bytes < plan.bytes || !aligned(workspace, 256))
    return SINKATTN_EWORKSPACE;
  const int64_t T = 128 / G;
  const int64_t dq_tiles = (int64_t(max_seqlen) + T - 1) / T;
  const int64_t kv_blocks = (int64_t(max_seqlen) + sa::kKvBN - 1) / sa::kKvBN;
  if (int64_t(batch) * num_kv_heads * dq_tiles > INT32_MAX) return SINKATTN_EUNSUPPORTED;

  sa::BwdArgs b;
  std::memset(&b, 0, sizeof b);
  b.Hq = num_q_heads;
  b.Hkv = num_kv_heads;
  b.G = G;
  b.batch = batch;
  b.total = total;
  b.window = window;
  b.rope_on = a.rope_on;
  b.rope_style = a.rope_style;
  b.scale_log2 = a.scale_log2;
  b.scale = static_cast<float>(static_cast<double>(a.scale_log2) / 1.4426950408889634);
  b.cu_seqlens = cu_seqlens;
  b.sink = sink;
  b.q = static_cast<const __nv_bfloat16 *>(q);
  b.k = static_cast<const __nv_bfloat16 *>(k);
  b.out = static_cast<const __nv_bfloat16 *>(out);
  b.dout = static_cast<const __nv_bfloat16 *>(dout);
  b.lse = lse;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  b.q_rot = reinterpret_cast<__nv_bfloat16 *>(ws + plan.q_rot);
  b.k_rot = reinterpret_cast<__nv_bfloat16 *>(ws + plan.k_rot);
  b.D = reinterpret_cast<float *>(ws + plan.D);
  b.dsink_part = reinterpret_cast<float *>(ws + plan.part);
  b.n_chunks = plan.chunks;
  b.dq = static_cast<__nv_bfloat16 *>(dq);
  b.dk = static_cast<__nv_bfloat16 *>(dk);
  b.dv = static_cast<__nv_bfloat16 *>(dv);
  b.dsink = dsink;
  b.dq_tiles = static_cast<int32_t>(dq_tiles);
  b.dq_items = static_cast<int32_t>(int64_t(batch) * num_kv_heads * dq_tiles);
  b.kv_blocks = static_cast<int32_t>(kv_blocks);
  b.kv_items = static_cast<int32_t>(int64_t(batch) * num_kv_heads * kv_blocks);
  b.grad_v8 = aligned(dq, 32) && aligned(dk, 32) && aligned(dv, 32) ? 1 : 0;
  std::memcpy(b.rope_turns, a.rope_turns, sizeof b.rope_turns);

  DeviceInfo dev;
  if (!device_info(dev)) return SINKATTN_ECUDA;
  if (dev.major != 10 || dev.minor != 3) return SINKATTN_EUNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  sa::bwd_pre_kernel<<<static_cast<unsigned>(plan.chunks), 256, 0, s>>>(b);
  if (cudaGetLastError() != cudaSuccess) return SINKATTN_ECUDA;
  sa::bwd_dsink_kernel<<<static_cast<unsigned>(num_q_heads), 256, 0, s>>>(b);
  if (cudaGetLastError() != cudaSuccess) return SINKATTN_ECUDA;

  // Q and K tiles: dims 0..63 from the rotated copies (from q and k as they
  // are without RoPE), dims 64..191 from q and k.
  CUtensorMap mq, mq0, mdo, mk, mk0, mv;
  auto qk_maps = [&](uint32_t q_rows, uint32_t k_rows) {
    if (!make_map(&mq, q, 192, num_q_heads, total, G, q_rows) ||
        !make_map(&mk, k, 192, num_kv_heads, total, 1, k_rows))
      return false;
    if (!a.rope_on) {
      mq0 = mq;
      mk0 = mk;
      return true;
    }
    return make_map(&mq0, b.q_rot, 64, num_q_heads, total, G, q_rows) &&
           make_map(&mk0, b.k_rot, 64, num_kv_heads, total, 1, k_rows);
  };
  // dq kernel: 128 packed rows (G heads x 128/G tokens) and 64-key blocks
  if (!qk_maps(static_cast<uint32_t>(T), sa::kDqBN) ||
      !make_map(&mdo, dout, 128, num_q_heads, total, G, static_cast<uint32_t>(T)) ||
      !make_map(&mv, v, 128, num_kv_heads, total, 1, sa::kDqBN))
    return SINKATTN_ECUDA;
  {
    auto kern = sa::bwd_dq_kernel;
    if (sinkattn_status st = smem_attr_once(kern, sa::DqLayout::kDynSmem)) return st;
    const int grid = static_cast<int>(std::min<int64_t>(b.dq_items, dev.sms));
    kern<<<grid, sa::kBwdThreads, sa::DqLayout::kDynSmem, s>>>(mq, mq0, mdo, mk, mk0, mv, b);
    if (sinkattn_status st = launched(kern)) return st;
  }
  // dkdv kernel: 64 packed rows (G heads x 64/G tokens) and 128-key blocks
  if (!qk_maps(static_cast<uint32_t>(sa::kKvRows / G), sa::kKvBN) ||
      !make_map(&mdo, dout, 128, num_q_heads, total, G, static_cast<uint32_t>(sa::kKvRows / G)) ||
      !make_map(&mv, v, 128, num_kv_heads, total, 1, sa::kKvBN))
    return SINKATTN_ECUDA;
  {
    auto kern = sa::bwd_dkdv_kernel;
    if (sinkattn_status st = smem_attr_once(kern, sa::KvLayout::kDynSmem)) return st;
    const int grid = static_cast<int>(std::min<int64_t>(b.kv_items, dev.sms));
    kern<<<grid, sa::kBwdThreads, sa::KvLayout::kDynSmem, s>>>(mq, mq0, mdo, mk, mk0, mv, b);
    if (sinkattn_status st = launched(kern)) return st;
  }
  return SINKATTN_OK;
}

const char *sinkattn_status_string(sinkattn_status s) {
  switch (s) {
    case SINKATTN_OK: return "ok";
    case SINKATTN_EINVAL: return "invalid argument";
    case SINKATTN_EUNSUPPORTED: return "unsupported shape or device";
    case SINKATTN_EWORKSPACE: return "workspace missing or too small";
    case SINKATTN_ECUDA: return "CUDA error";
    case SINKATTN_ETIMEOUT: return "kernel wait timed out";
    case SINKATTN_ECHECK: return "bounds check failed (checking build)";
  }
  return "unknown status";
}

sinkattn_status sinkattn_get_device_status(uint32_t *detail) {
  if (cudaDeviceSynchronize() != cudaSuccess) return SINKATTN_ECUDA;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbol(&word, sa::g_status_word, sizeof word) != cudaSuccess)
    return SINKATTN_ECUDA;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(sa::g_status_word, &zero, sizeof zero) != cudaSuccess)
    return SINKATTN_ECUDA;
  if (detail) *detail = word;
  if (word & 1u) return SINKATTN_ETIMEOUT;
  return (word & 2u) ? SINKATTN_ECHECK : SINKATTN_OK;
}

sinkattn_status sinkattn_prefill_ex(const void *q, const void *k, const void *v, const float *sink,
                                    const int32_t *cu_seqlens, int32_t batch, int32_t total,
                                    int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t window, float rope_base, const sinkattn_params *params,
                                    void *out, float *lse, sinkattn_stream_t stream) {
  // ------------------------------------------------ host-side checks (no CUDA call)
  if (batch < 0 || total < 0 || max_seqlen < 0 || window < 0) return SINKATTN_EINVAL;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return SINKATTN_EINVAL;
  if (!pow2_upto_128(num_q_heads / num_kv_heads)) return SINKATTN_EUNSUPPORTED;
  if (num_q_heads > 65535 || num_kv_heads > 65535) return SINKATTN_EUNSUPPORTED;
  if (total > 0 && max_seqlen == 0) return SINKATTN_EINVAL;
  if (batch == 0 || total == 0) return SINKATTN_OK;
  if (!q || !k || !v || !sink || !cu_seqlens || !out || !lse) return SINKATTN_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(sink, 4) || !aligned(cu_seqlens, 4))
    return SINKATTN_EINVAL;
  AttnArgs a;
  // a prefill reads no cache: neither a ring nor pre-rotated keys
  if (params && (params->kv_ring || params->k_rotated)) return SINKATTN_EINVAL;
  if (sinkattn_status st = fill_common(a, params, rope_base, num_q_heads, num_kv_heads, window))
    return st;

  // ------------------------------------------------ schedule
  const int32_t G = a.G;
  const int32_t tile_tokens = 128 / G;
  // Sliding windows that fit one 144-key block per tile take the single-block
  // kernel; global or wide windows take the multi-block online-softmax kernel.
  const bool wide = window > 0 && window + tile_tokens - 1 <= kBNWide;
  const int32_t BN = wide ? kBNWide : kBN;
  a.batch = batch;
  a.tile_tokens = tile_tokens;
  a.tiles_per_seq = (max_seqlen + tile_tokens - 1) / tile_tokens;
  const int64_t n_items = int64_t(batch) * num_kv_heads * a.tiles_per_seq;
  if (n_items > INT32_MAX) return SINKATTN_EUNSUPPORTED;
  a.n_items = static_cast<int32_t>(n_items);
  a.lpt_order = window == 0 ? 1 : 0;
  a.q_tx_bytes = 3u * 64u * 2u * static_cast<uint32_t>(G * tile_tokens);
  a.cu_seqlens = cu_seqlens;
  a.sink = sink;
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.lse = lse;
  a.n_rows = int64_t(total) * num_q_heads;

  DeviceInfo dev;
  if (!device_info(dev)) return SINKATTN_ECUDA;
  if (dev.major != 10 || dev.minor != 3) return SINKATTN_EUNSUPPORTED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (G == sa::kBandG && window >= 1 && window <= sa::kBandMaxWin * sa::kBandSeg - sa::kBandSeg &&
      a.scale_log2 > 0.f)
    return launch_band(q, k, v, a, cu_seqlens, batch, total, dev, s);
  // every other shape, global or windowed: the two-tile causal kernel (a
  // window only trims the key blocks of an item)
  if (a.scale_log2 > 0.f)
    return launch_causal(q, k, v, a, cu_seqlens, batch, total, max_seqlen, dev, s);
  // a logit scale <= 0: the general kernel (the band and causal kernels take
  // the maximum of the raw logits and scale it, which is the maximum of the
  // scaled logits only for a positive scale)

  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, 192, num_q_heads, total, G, tile_tokens) ||
      !make_map(&mk, k, 192, num_kv_heads, total, 1, BN) ||
      !make_map(&mv, v, 128, num_kv_heads, total, 1, BN))
    return SINKATTN_ECUDA;
  const int grid = static_cast<int>(std::min<int64_t>(n_items, dev.sms));
  if (wide) return launch<kBNWide, 2, 1>(mq, mk, mv, a, grid, s);
  return launch<kBN, 1, 2>(mq, mk, mv, a, grid, s);
}

sinkattn_status sinkattn_prefill(const void *q, const void *k, const void *v, const float *sink,
                                 const int32_t *cu_seqlens, int32_t batch, int32_t total,
                                 int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t window, float rope_base, void *out, float *lse,
                                 sinkattn_stream_t stream) {
  return sinkattn_prefill_ex(q, k, v, sink, cu_seqlens, batch, total, max_seqlen, num_q_heads,
                             num_kv_heads, window, rope_base, nullptr, out, lse, stream);
}

size_t sinkattn_decode_workspace_size(int32_t batch, int32_t T, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t max_seqlen, int32_t window) {
  if (batch <= 0 || T <= 0 || max_seqlen < 0 || window < 0) return 0;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  const int32_t G = num_q_heads / num_kv_heads;
  if (!pow2_upto_128(G) || T * G > 128) return 0;
  return decode_plan(batch, T, num_q_heads, num_kv_heads).bytes;
}

// A 3-D tensor map over rows of `heads` x `dim_bytes` E4M3 bytes: dims
// (dim_bytes, heads, rows), a box of one head's whole row x box_rows, no swizzle
// (the conversion warps read it as plain rows).
bool make_map_u8(CUtensorMap *m, const void *base, uint64_t dim_bytes, uint64_t heads, uint64_t rows,
                 uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t gdim[3] = {dim_bytes, heads, rows};
  const cuuint64_t gstride[2] = {dim_bytes, dim_bytes * heads};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(dim_bytes), 1, box_rows};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), gdim, gstride,
                        box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Shared by the bf16 and the FP8 decode (k_scale != nullptr: the cache holds
// E4M3 values, dequantised as value * scale[kv head]).
static sinkattn_status decode_impl(const void *q, const void *kcache, const void *vcache,
                                   const int32_t *seqlens, const float *sink, int32_t window,
                                   float rope_base, int32_t batch, int32_t T, int32_t S_cap,
                                   int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                   const sinkattn_params *params, void *workspace,
                                   size_t workspace_bytes, void *out, float *lse,
                                   sinkattn_stream_t stream, const float *k_scale,
                                   const float *v_scale) {
  const bool fp8 = k_scale != nullptr;
  if (batch < 0 || T <= 0 || S_cap <= 0 || max_seqlen < 0 || window < 0) return SINKATTN_EINVAL;
  const bool ring = params && params->kv_ring;
  const bool k_rotated = params && params->k_rotated;
  if (params && params->kv_ring != 0 && params->kv_ring != 1) return SINKATTN_EINVAL;
  if (params && params->k_rotated != 0 && params->k_rotated != 1) return SINKATTN_EINVAL;
  if (ring) {
    // the visible positions [L - T - W + 1, L) must sit in distinct slots, read
    // in 16-key pieces that never straddle the ring's end
    if (window <= 0 || int64_t(S_cap) < int64_t(window) + T - 1 || S_cap % 16) return SINKATTN_EINVAL;
  } else if (max_seqlen > S_cap) {
    return SINKATTN_EINVAL;
  }
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return SINKATTN_EINVAL;
  const int32_t G = num_q_heads / num_kv_heads;
  if (!pow2_upto_128(G)) return SINKATTN_EUNSUPPORTED;
  if (T * G > 128) return SINKATTN_EUNSUPPORTED;
  if (int64_t(batch) * S_cap > INT32_MAX || int64_t(batch) * T > INT32_MAX)
    return SINKATTN_EUNSUPPORTED;
  if (batch == 0) return SINKATTN_OK;
  if (!q || !kcache || !vcache || !seqlens || !sink || !out || !lse) return SINKATTN_EINVAL;
  if (fp8 && (ring || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4))) return SINKATTN_EINVAL;
  if (!aligned(q, 16) || !aligned(kcache, 16) || !aligned(vcache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(sink, 4) || !aligned(seqlens, 4))
    return SINKATTN_EINVAL;
  const DecodePlan plan = decode_plan(batch, T, num_q_heads, num_kv_heads);
  if (!workspace || workspace_bytes < plan.bytes || !aligned(workspace, 256))
    return SINKATTN_EWORKSPACE;
  AttnArgs a;
  if (sinkattn_status st = fill_common(a, params, rope_base, num_q_heads, num_kv_heads, window))
    return st;
  if (!(a.scale_log2 > 0.f)) return SINKATTN_EINVAL;  // the decode softmax scales after the max
  if (int64_t(batch) * num_kv_heads > INT32_MAX / 2) return SINKATTN_EUNSUPPORTED;

  sa::DecArgs d;
  std::memset(&d, 0, sizeof d);
  d.Hq = num_q_heads;
  d.Hkv = num_kv_heads;
  d.G = G;
  d.T = T;
  d.R = plan.rows;
  d.window = window;
  d.batch = batch;
  d.S_cap = S_cap;
  d.n_units = batch * num_kv_heads;
  d.kv_ring = ring ? 1 : 0;
  d.k_rotated = k_rotated ? 1 : 0;
  d.k_scale = k_scale;
  d.v_scale = v_scale;
  d.rope_on = a.rope_on;
  d.rope_style = a.rope_style;
  d.q_tx_bytes = 3u * 64u * 2u * static_cast<uint32_t>(G * T);
  d.scale_log2 = a.scale_log2;
  d.seqlens = seqlens;
  d.sink = sink;
  d.out = static_cast<__nv_bfloat16 *>(out);
  d.lse = lse;
  d.tickets = static_cast<unsigned long long *>(workspace);
  d.epoch = next_decode_epoch();
  d.part_o = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + plan.tab_bytes);
  d.part_ml = d.part_o + static_cast<size_t>(sa::kDecMaxGrid) * 2 * plan.rows * sa::kDv;
  d.n_rows = int64_t(batch) * T * num_q_heads;
  d.n_part_rows = int64_t(sa::kDecMaxGrid) * 2 * plan.rows;
  std::memcpy(d.rope_turns, a.rope_turns, sizeof d.rope_turns);

  DeviceInfo dev;
  if (!device_info(dev)) return SINKATTN_ECUDA;
  if (dev.major != 10 || dev.minor != 3) return SINKATTN_EUNSUPPORTED;

  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, 192, num_q_heads, uint64_t(batch) * T, G, T) ||
      (fp8 ? !make_map_u8(&mk, kcache, 192, num_kv_heads, uint64_t(batch) * S_cap, sa::kDecBN)
           : !make_map(&mk, kcache, 192, num_kv_heads, uint64_t(batch) * S_cap, 1,
                       ring ? 16 : sa::kDecBN)) ||
      (fp8 ? !make_map_u8(&mv, vcache, 128, num_kv_heads, uint64_t(batch) * S_cap, sa::kDecBN)
           : !make_map(&mv, vcache, 128, num_kv_heads, uint64_t(batch) * S_cap, 1,
                       ring ? 16 : sa::kDecBN)))
    return SINKATTN_ECUDA;
  // upper bound of the blocks: every unit sees at most max_seqlen (window: T + W - 1) keys,
  // plus up to 15 before them when a ring cache aligns its first block
  const int64_t range = window > 0 ? std::min<int64_t>(max_seqlen, int64_t(T) + window - 1 + (ring ? 15 : 0))
                                   : int64_t(max_seqlen);
  // one block list per KV head (its CTAs walk the sequences' cache rows with
  // the other heads' CTAs) unless there are more KV heads than CTAs
  const int cap = std::min<int>(dev.sms, sa::kDecMaxGrid);
  d.n_sub = num_kv_heads <= cap ? num_kv_heads : 1;
  d.n_k = d.n_units / d.n_sub;
  const int64_t max_blocks = int64_t(d.n_k) * ((range + sa::kDecBN - 1) / sa::kDecBN);
  const int groups = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(max_blocks, cap / d.n_sub)));
  const int grid = groups * d.n_sub;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fp8) {
    auto kern = sa::sinkattn_decode_kernel<true>;
    constexpr uint32_t smem = sa::DecLayoutT<true>::kDynSmem;
    if (sinkattn_status st = smem_attr_once(kern, smem)) return st;
    kern<<<grid, sa::DecThreads<true>::kAll, smem, s>>>(mq, mk, mv, d);
    return launched(kern);
  } else {
    auto kern = sa::sinkattn_decode_kernel<false>;
    constexpr uint32_t smem = sa::DecLayoutT<false>::kDynSmem;
    if (sinkattn_status st = smem_attr_once(kern, smem)) return st;
    kern<<<grid, sa::kThreads, smem, s>>>(mq, mk, mv, d);
    return launched(kern);
  }
}

sinkattn_status sinkattn_decode_ex(const void *q, const void *kcache, const void *vcache,
                                   const int32_t *seqlens, const float *sink, int32_t window,
                                   float rope_base, int32_t batch, int32_t T, int32_t S_cap,
                                   int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                   const sinkattn_params *params, void *workspace,
                                   size_t workspace_bytes, void *out, float *lse,
                                   sinkattn_stream_t stream) {
  return decode_impl(q, kcache, vcache, seqlens, sink, window, rope_base, batch, T, S_cap,
                     max_seqlen, num_q_heads, num_kv_heads, params, workspace, workspace_bytes,
                     out, lse, stream, nullptr, nullptr);
}

sinkattn_status sinkattn_decode_fp8(const void *q, const void *kcache, const void *vcache,
                                    const float *k_scale, const float *v_scale,
                                    const int32_t *seqlens, const float *sink, int32_t window,
                                    float rope_base, int32_t batch, int32_t T, int32_t S_cap,
                                    int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                    const sinkattn_params *params, void *workspace,
                                    size_t workspace_bytes, void *out, float *lse,
                                    sinkattn_stream_t stream) {
  if (!k_scale || !v_scale) return SINKATTN_EINVAL;
  return decode_impl(q, kcache, vcache, seqlens, sink, window, rope_base, batch, T, S_cap,
                     max_seqlen, num_q_heads, num_kv_heads, params, workspace, workspace_bytes,
                     out, lse, stream, k_scale, v_scale);
}

sinkattn_status sinkattn_decode(const void *q, const void *kcache, const void *vcache,
                                const int32_t *seqlens, const float *sink, int32_t window,
                                float rope_base, int32_t batch, int32_t T, int32_t S_cap,
                                int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                void *workspace, size_t workspace_bytes, void *out, float *lse,
                                sinkattn_stream_t stream) {
  return sinkattn_decode_ex(q, kcache, vcache, seqlens, sink, window, rope_base, batch, T, S_cap,
                            max_seqlen, num_q_heads, num_kv_heads, nullptr, workspace,
                            workspace_bytes, out, lse, stream);
}

}  // extern "C"

// ------------------------------------------------------------------------------
// Decode without any allocation by the caller or the library.
//
// Some callers cannot allocate device memory at the point where they run
// decode: code inside an allocator-free region (a memory pool that must not
// grow, a real-time path that forbids cudaMalloc and its implicit
// synchronisation), or a host that owns no device allocator at all.  For them,
// the split-KV partials live in one fixed buffer that is part of the library's
// own device image: every GPU that loads the library holds these
// SINKATTN_NOALLOC_SCRATCH_BYTES until the process exits.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SINKATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device, looked up once per
// device (host code only sees a host-side stand-in for the symbol).
sinkattn_status noalloc_scratch(void **ptr) {
  static std::mutex mu;
  static void *addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SINKATTN_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return SINKATTN_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SINKATTN_ECUDA;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return SINKATTN_OK;
}

}  // namespace

extern "C" sinkattn_status sinkattn_decode_noalloc(
    const void *q, const void *kcache, const void *vcache, const int32_t *seqlens,
    const float *sink, int32_t window, float rope_base, int32_t batch, int32_t T, int32_t S_cap,
    int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads, void *out, float *lse,
    sinkattn_stream_t stream) {
  const size_t need =
      sinkattn_decode_workspace_size(batch, T, num_q_heads, num_kv_heads, max_seqlen, window);
  if (need > SINKATTN_NOALLOC_SCRATCH_BYTES) return SINKATTN_EWORKSPACE;
  // need == 0: an empty batch (nothing to do) or arguments sinkattn_decode
  // rejects; either way it answers before any CUDA call, and the scratch
  // buffer is not looked up.
  if (need == 0) return sinkattn_decode(q, kcache, vcache, seqlens, sink, window, rope_base, batch,
                                        T, S_cap, max_seqlen, num_q_heads, num_kv_heads, nullptr,
                                        0, out, lse, stream);
  void *scratch = nullptr;
  if (sinkattn_status st = noalloc_scratch(&scratch)) return st;
  // Every partial a merge reads is written first by the same call, and the
  // tickets carry the call's own number, so the buffer needs no clearing.
  return sinkattn_decode(q, kcache, vcache, seqlens, sink, window, rope_base, batch, T, S_cap,
                         max_seqlen, num_q_heads, num_kv_heads, scratch,
                         SINKATTN_NOALLOC_SCRATCH_BYTES, out, lse, stream);
}

#ifdef SINKATTN_TEST_HOOKS
// Test builds only: see sa::g_test_stall_ns.  0 turns the stall off.
extern "C" int sinkattn_test_set_stall_ns(uint64_t ns) {
  return cudaMemcpyToSymbol(sa::g_test_stall_ns, &ns, sizeof ns) == cudaSuccess ? 0 : 1;
}
#endif

#ifdef SINKATTN_CHECKS
// Checking builds only: make the checks see every tensor as `row_shrink` rows
// (or elements) shorter and admit only `tmem_cols` TMEM columns, so a test can
// see them fire without any access actually out of bounds.  (0, 512) restores
// the true limits.
extern "C" int sinkattn_test_set_check_limits(int64_t row_shrink, uint32_t tmem_cols) {
  if (row_shrink < 0 || tmem_cols > 512) return 1;
  if (cudaMemcpyToSymbol(sa::g_check_row_shrink, &row_shrink, sizeof row_shrink) != cudaSuccess)
    return 1;
  return cudaMemcpyToSymbol(sa::g_check_tmem_cols, &tmem_cols, sizeof tmem_cols) == cudaSuccess
             ? 0 : 1;
}
#endif
