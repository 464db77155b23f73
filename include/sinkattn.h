/*
 * sinkattn.h -- C ABI of the sink-bias GQA attention forward pass for B300 (sm_103a).
 *
 * The operation is the attention layer of the "MiMo-V2-Flash Technical Report"
 * (full Chinese translation, garden.houmin.site/digest/mimo-v2-flash):
 *
 *   §2.2 eq. (1)  a_ij = q_i . k_j / sqrt(d)          (d = 192, the QK head dim)
 *   §2.2 eq. (2)  s_ij = exp(a_ij - m_i) / (exp(sink_h - m_i) + sum_j' exp(a_ij' - m_i)),
 *                 m_i = max(max_j a_ij, sink_h)      (one learnable sink per query head)
 *   §2.2 eq. (3)  o_i = sum_j s_ij v_j                (the sink carries no value)
 *
 * with the shapes of §2.1 Table 1: grouped-query attention (SWA layers 64 query /
 * 8 KV heads with a 128-token sliding window; GA layers 64 query / 4 KV heads,
 * global causal), QK head dim 192, V head dim 128, and rotary position
 * embedding on the first 64 dims of q and k only (RoPE base 10,000 for SWA,
 * 5,000,000 for GA after the 256K extension, §3.2).
 *
 * Conventions shared by every call:
 *   - All tensor arguments are DEVICE pointers owned by the caller, dense and
 *     row-major with the head index varying faster than the token index.
 *     q, k, v, kcache, vcache and out must be 16-byte aligned; lse and sink
 *     4-byte aligned.  The library keeps no pointer after a call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  No call allocates, frees or synchronises, except
 *     sinkattn_get_device_status, which synchronises the current device.
 *   - Window: window = 0 means global causal attention; window = W > 0 means key
 *     j is visible to query i iff i - W < j <= i (W keys including i itself).
 *   - Keys are passed UNROTATED; the kernels rotate q and k on chip.  RoPE pairs
 *     dims (2t, 2t+1) for t < 32 with angle pos * base^(-2t/64) (RoFormer), unless
 *     a params struct selects pairs (t, t+32).
 *   - Input range of the rotated dims.  The forward kernels keep dims 0..63 of
 *     q and k, after the rotation, as fp16 (11 significant bits instead of
 *     bf16's 8).  A rotation keeps the length of each pair, so every rotated
 *     pair (x, y) of q and k must have sqrt(x^2 + y^2) <= 65504 (guaranteed when
 *     |x|, |y| <= 46000); a longer pair overflows to inf and its rows come out
 *     NaN, with no status.  Values below 2^-14 (about 6.1e-5) are kept as fp16
 *     subnormals, with an absolute step of 2^-24 (about 6e-8).  The FP8-cache
 *     decode also rounds dims 64..191 of q to fp16 (|q| <= 65504 there).  The
 *     backward pass keeps bf16 copies and has no such limit.
 *   - lse is the natural-log log-sum-exp of the row INCLUDING the sink:
 *     lse_i = ln(exp(sink_h) + sum_{j visible} exp(a_ij)).
 *   - out is bf16 (round to nearest even of the fp32 result), lse fp32.
 *   - A row with no visible key gets out = 0 and lse = sink (-inf if the sink
 *     is -inf).
 *   - Functions return a status and never throw.  SINKATTN_EINVAL and
 *     SINKATTN_EUNSUPPORTED are returned before anything is launched;
 *     SINKATTN_ECUDA reports a CUDA error from a launch; kernels that hit an
 *     internal wait limit record SINKATTN_ETIMEOUT in a device status word
 *     that sinkattn_get_device_status reads.  Kernels never trap.
 *   - A build with -DSINKATTN_CHECKS (the test library) also checks, inside
 *     the kernels, every TMA copy's x coordinate and shared-memory
 *     destination, every TMEM access and MMA operand, and every global store
 *     index against its tensor's extent; a failed check skips that access and
 *     records SINKATTN_ECHECK.  The product library carries no checks.
 *   - Results are deterministic: the same inputs give the same bits.
 */
#ifndef SINKATTN_H
#define SINKATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SINKATTN_OK = 0,
    SINKATTN_EINVAL = 1,       /* bad pointer, size, alignment or combination */
    SINKATTN_EUNSUPPORTED = 2, /* head dims, group size or device not supported */
    SINKATTN_EWORKSPACE = 3,   /* decode workspace missing or too small */
    SINKATTN_ECUDA = 4,        /* a CUDA runtime call failed */
    SINKATTN_ETIMEOUT = 5,     /* a kernel gave up on an internal wait */
    SINKATTN_ECHECK = 6        /* a bounds check failed (checking builds only) */
} sinkattn_status;

/* cudaStream_t, passed as an opaque pointer so that this header needs no CUDA include. */
typedef void *sinkattn_stream_t;

/* Optional knobs of the _ex calls.  Zero-initialise for the defaults. */
typedef struct {
    float scale;        /* logit scale; 0 -> 1/sqrt(192) (eq. (1) with d = 192) */
    int32_t rope_off;   /* 1 -> no rotary embedding at all (positions ignored) */
    int32_t rope_style; /* 0 -> pairs (2t, 2t+1) (default); 1 -> pairs (t, t+32) */
    int32_t kv_ring;    /* decode only (prefill rejects it): 1 -> kcache/vcache are rings of
                           S_cap slots holding the latest keys, position j at slot j % S_cap
                           (the KV cache of a sliding-window layer keeps only its window) */
    int32_t k_rotated;  /* decode only (prefill and backward reject it): 1 -> kcache holds
                           every key already rotated at its own absolute position (a
                           serving cache that stores keys after RoPE), so the decode
                           rotates only q.  With a bf16 cache the rotated dims of q are
                           then kept in bf16 (the cache's type) instead of fp16 */
} sinkattn_params;

/*
 * Prefill over a varlen batch of self-attention sequences (the forward pass of
 * one SWA or GA layer, §2.1-§2.2).
 *
 *   q          bf16 [total, num_q_heads, 192]
 *   k          bf16 [total, num_kv_heads, 192], unrotated
 *   v          bf16 [total, num_kv_heads, 128]
 *   sink       fp32 [num_q_heads], may hold -inf (no sink for that head)
 *   cu_seqlens int32 [batch + 1], device: cu_seqlens[0] = 0, non-decreasing,
 *              cu_seqlens[batch] = total.  Sequence b holds tokens
 *              cu_seqlens[b] .. cu_seqlens[b+1]-1 at RoPE positions 0, 1, ...
 *   batch, total, max_seqlen  host copies of the sizes; max_seqlen must be at
 *              least the longest sequence (it bounds the tile schedule).
 *   num_q_heads / num_kv_heads  must be a power of two between 1 and 128;
 *              query head h uses KV head h / (num_q_heads / num_kv_heads).
 *   window     0 = global causal, W > 0 = sliding window of W keys.
 *   rope_base  RoPE base (> 0).
 *   out        bf16 [total, num_q_heads, 128]
 *   lse        fp32 [total, num_q_heads]
 */
sinkattn_status sinkattn_prefill(const void *q, const void *k, const void *v, const float *sink,
                                 const int32_t *cu_seqlens, int32_t batch, int32_t total,
                                 int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t window, float rope_base, void *out, float *lse,
                                 sinkattn_stream_t stream);

sinkattn_status sinkattn_prefill_ex(const void *q, const void *k, const void *v, const float *sink,
                                    const int32_t *cu_seqlens, int32_t batch, int32_t total,
                                    int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t window, float rope_base, const sinkattn_params *params,
                                    void *out, float *lse, sinkattn_stream_t stream);

/*
 * Bytes of device workspace sinkattn_decode needs for these sizes.  The decode
 * cuts every unit's (sequence, KV head) visible keys into 64-key blocks and
 * splits the list of all blocks evenly over at most 160 CTAs, in one launch.
 * A unit a CTA boundary cuts leaves, per CTA, its running max, sum and
 * unnormalised output without the sink; the CTA that finishes the unit last
 * (told by the unit's ticket) merges them and adds the sink once.  The
 * workspace holds one 64-bit ticket per unit (batch * num_kv_heads, padded to
 * 256 bytes) and, per CTA, two partial slots of T * (num_q_heads /
 * num_kv_heads) rows x 132 fp32 (§2.3.1's multi-token verify split over the
 * cache).  It does not depend on the cache lengths or the window.  Returns 0
 * for arguments sinkattn_decode would reject.
 */
size_t sinkattn_decode_workspace_size(int32_t batch, int32_t T, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t max_seqlen, int32_t window);

/*
 * Multi-token (MTP-verify) decode against a KV cache (§2.3.1: the main model
 * verifies 1 + K draft tokens in one pass without extra KV-cache I/O).  The T
 * new tokens of each sequence are already appended to the cache.
 *
 *   q        bf16 [batch, T, num_q_heads, 192]; query t of sequence b sits at
 *            position seqlens[b] - T + t and sees cache positions j <= its own
 *            position (causal among the drafts) and, with a window, j > pos - W.
 *   kcache   bf16 [batch, S_cap, num_kv_heads, 192], unrotated keys at positions 0..
 *   vcache   bf16 [batch, S_cap, num_kv_heads, 128]
 *   seqlens  int32 [batch], device: cached tokens including the T new ones,
 *            T <= seqlens[b] <= S_cap (shorter caches give empty rows).  Cache
 *            rows at or past seqlens[b] are never used and may hold anything.
 *   max_seqlen  host bound on max(seqlens).
 *   T        1 <= T and T * (num_q_heads / num_kv_heads) <= 128.
 *   workspace, workspace_bytes  device scratch of at least
 *            sinkattn_decode_workspace_size(...) bytes, 256-byte aligned; it
 *            needs no clearing (each call's tickets carry a number of their
 *            own) and its contents are rewritten by every call.  Calls that
 *            share one workspace must not overlap on the GPU.
 *   The logit scale must be positive (sinkattn_decode_ex with a scale <= 0
 *   returns SINKATTN_EINVAL).
 *   Ring cache (sinkattn_decode_ex with params->kv_ring = 1; the KV cache of an
 *   SWA layer, §2.1: only the window is ever read): kcache/vcache hold S_cap
 *   slots per sequence and the key at position j sits at slot j % S_cap, so
 *   seqlens[b] may exceed S_cap.  Positions keep their absolute values for
 *   RoPE and the mask.  Requires window > 0, S_cap >= window + T - 1 (the T
 *   queries see the last window + T - 1 positions) and S_cap a multiple of 16;
 *   otherwise SINKATTN_EINVAL.  Slots outside the visible positions may hold
 *   anything.
 *   out      bf16 [batch, T, num_q_heads, 128];  lse fp32 [batch, T, num_q_heads]
 */
sinkattn_status sinkattn_decode(const void *q, const void *kcache, const void *vcache,
                                const int32_t *seqlens, const float *sink, int32_t window,
                                float rope_base, int32_t batch, int32_t T, int32_t S_cap,
                                int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                void *workspace, size_t workspace_bytes, void *out, float *lse,
                                sinkattn_stream_t stream);

sinkattn_status sinkattn_decode_ex(const void *q, const void *kcache, const void *vcache,
                                   const int32_t *seqlens, const float *sink, int32_t window,
                                   float rope_base, int32_t batch, int32_t T, int32_t S_cap,
                                   int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                   const sinkattn_params *params, void *workspace,
                                   size_t workspace_bytes, void *out, float *lse,
                                   sinkattn_stream_t stream);

/*
 * MTP-verify decode over an FP8 KV cache.  The report trains and serves in FP8
 * (§4.6: training and inference both run FP8) but gives no scale convention;
 * here the cache holds E4M3 values with one fp32 scale per KV head for K and
 * one for V (the key is e4m3 * k_scale[kv head], the value e4m3 * v_scale).
 *   kcache   E4M3 bytes [batch, S_cap, num_kv_heads, 192], unrotated keys
 *   vcache   E4M3 bytes [batch, S_cap, num_kv_heads, 128]
 *   k_scale, v_scale  fp32 [num_kv_heads], device
 * Everything else as sinkattn_decode_ex (same workspace size); params->kv_ring
 * must be 0.  The cache rows are converted to fp16 on chip (exactly) and the
 * keys rotated there; q is rounded to fp16 and the products run fp16 x fp16
 * with fp32 accumulation.  The cache read is half the bf16 cache's.
 */
sinkattn_status sinkattn_decode_fp8(const void *q, const void *kcache, const void *vcache,
                                    const float *k_scale, const float *v_scale,
                                    const int32_t *seqlens, const float *sink, int32_t window,
                                    float rope_base, int32_t batch, int32_t T, int32_t S_cap,
                                    int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                                    const sinkattn_params *params, void *workspace,
                                    size_t workspace_bytes, void *out, float *lse,
                                    sinkattn_stream_t stream);

/*
 * sinkattn_decode_noalloc -- sinkattn_decode for callers that cannot allocate.
 *
 * This entry point has no counterpart in the report; it exists for callers that
 * must not allocate device memory when they decode (an allocator-free region,
 * a fixed memory pool that may not grow, a host without a device allocator).  It takes the same arguments as sinkattn_decode
 * minus the workspace: the split-KV partials go to one fixed buffer of
 * SINKATTN_NOALLOC_SCRATCH_BYTES that is part of the library's device image, so
 * every GPU that loads the library holds that memory until the process exits.
 * Nothing is allocated or freed by this call.
 *
 *   - Sizes whose partials need more than SINKATTN_NOALLOC_SCRATCH_BYTES (see
 *     sinkattn_decode_workspace_size) are rejected with SINKATTN_EWORKSPACE
 *     before anything is launched.
 *   - The first call on each device looks up the buffer's device address
 *     (cudaGetSymbolAddress on that device) and keeps it for the life of the
 *     process; make that first call before any stream capture.  A
 *     cudaDeviceReset (or anything else that destroys the device's primary
 *     context) invalidates the kept address: do not call this entry point on
 *     that device afterwards.
 *   - Arguments sinkattn_decode would reject get the same status, before the
 *     buffer is looked up; an empty batch returns SINKATTN_OK.
 *   - All calls share the one buffer per device: calls that overlap on the GPU
 *     (other streams, other host threads) race and give wrong results.  Calls
 *     on one stream are ordered and safe.
 *   - The buffer keeps the previous call's contents; no call needs it cleared.
 */
#define SINKATTN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
sinkattn_status sinkattn_decode_noalloc(const void *q, const void *kcache, const void *vcache,
                                        const int32_t *seqlens, const float *sink, int32_t window,
                                        float rope_base, int32_t batch, int32_t T, int32_t S_cap,
                                        int32_t max_seqlen, int32_t num_q_heads,
                                        int32_t num_kv_heads, void *out, float *lse,
                                        sinkattn_stream_t stream);

/*
 * Backward pass of sinkattn_prefill (the sink logits are learned, §2.2; the
 * pages define the forward, eqs. (1)-(3), and this is its plain derivative for
 * the loss L = sum dout . out):
 *   dq, dk, dv  gradients of L with respect to q, k, v (raw, unrotated inputs)
 *   dsink       gradient with respect to sink: -sum_i exp(sink_h - lse_i) (dout_i . out_i)
 *
 *   q, k, v, sink, cu_seqlens, batch, total, max_seqlen, num_q_heads,
 *   num_kv_heads, window, rope_base, params   as for sinkattn_prefill_ex (params
 *              may be NULL; kv_ring must be 0)
 *   out, lse   the forward's outputs for these inputs (bf16 [total, Hq, 128],
 *              fp32 [total, Hq])
 *   dout       bf16 [total, num_q_heads, 128]
 *   workspace, workspace_bytes  device scratch of at least
 *              sinkattn_prefill_backward_workspace_size(...) bytes, 256-byte
 *              aligned; no clearing needed.  It holds the rotated q and k and
 *              the row terms dout_i . out_i.
 *   dq bf16 [total, Hq, 192], dk bf16 [total, Hkv, 192], dv bf16 [total, Hkv, 128],
 *   dsink fp32 [Hq]: all fully written.
 * Needs 1 <= num_q_heads / num_kv_heads <= 64 and a positive scale
 * (SINKATTN_EUNSUPPORTED / SINKATTN_EINVAL otherwise).  Deterministic.
 */
size_t sinkattn_prefill_backward_workspace_size(int32_t total, int32_t num_q_heads,
                                                int32_t num_kv_heads);
sinkattn_status sinkattn_prefill_backward(const void *q, const void *k, const void *v,
                                          const float *sink, const int32_t *cu_seqlens,
                                          int32_t batch, int32_t total, int32_t max_seqlen,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t window, float rope_base,
                                          const sinkattn_params *params, const void *out,
                                          const float *lse, const void *dout, void *workspace,
                                          size_t workspace_bytes, void *dq, void *dk, void *dv,
                                          float *dsink, sinkattn_stream_t stream);

/* A static string naming a status code. */
const char *sinkattn_status_string(sinkattn_status status);

/*
 * Synchronises the current device, then reads and clears the library's device
 * status word.  Returns SINKATTN_OK, SINKATTN_ETIMEOUT (a kernel gave up on a
 * wait and wrote no trustworthy output), SINKATTN_ECHECK (only a library built
 * with SINKATTN_CHECKS: an in-kernel bounds check failed and its access was
 * skipped) or SINKATTN_ECUDA.  `detail`, if not NULL, receives the raw word
 * (bit 0: timeout, bits 8..15: the wait site; bit 1: a failed check, bits
 * 16..23: the check site).
 */
sinkattn_status sinkattn_get_device_status(uint32_t *detail);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH.  0.2.0 added
 * sinkattn_params.k_rotated (the struct grew by one int32). */
int32_t sinkattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SINKATTN_H */
