/*
 * vc.h -- C ABI of the GB300 (sm_103a) hot path of VeriCache's lossless
 * draft -> verify -> accept decode loop.
 *
 * Source of the method: "VeriCache: Turning Lossy KV Cache into Lossless LLM
 * Inference" (gist.science/paper/2605.17613), Technical Summary:
 *   - Core Algorithm: draft with the compressed KV, verify with one forward
 *     pass over the full KV, accept up to the first mismatch (+ bonus token);
 *   - Key System Innovations (1): drafting is HBM-bound, verification is
 *     interconnect-bound; requests are staggered so the two overlap;
 *   - Architecture Support: compressed KV in GPU memory, full KV in CPU
 *     memory loaded over the CPU-GPU link for verification; a uniform
 *     compressor interface for token-dropping and quantisation methods
 *     (KIVI, SnapKV named).
 *
 * Five shared libraries implement this header:
 *   libvc_core.so         status strings, last-error text (used by the others)
 *   libvc_quant_kv.so     compressors: KIVI-style pack / append, SnapKV-style
 *                         score / select / gather
 *   libvc_draft_attn.so   decode attention over the packed draft cache
 *   libvc_verify_attn.so  verify attention over the full KV streamed from
 *                         pinned host memory, commit of accepted tokens
 *   libvc_accept.so       argmax / first-mismatch / bonus token
 *
 * Conventions (all entry points):
 *   - Every call returns vc_status_t.  Argument errors are detected on the
 *     host and returned before anything is launched; vc_last_error() then
 *     holds a one-line reason (thread-local).  No exception crosses the ABI.
 *   - Compute calls are asynchronous on the stream given (NULL = the legacy
 *     default stream).  A fault inside a kernel surfaces at the caller's next
 *     synchronisation.  Kernels that wait on a barrier give up after a bounded
 *     time and raise a device error flag, read with vc_*_device_status().
 *   - The caller owns every buffer (device memory, pinned host memory); the
 *     libraries allocate nothing per call.  Scratch space is passed in as a
 *     workspace whose size the *_workspace_size() query returns.
 *   - Pointers are plain addresses: "device" = memory the GPU can address
 *     (cudaMalloc / PyTorch CUDA tensors); "pinned host" = cudaHostAlloc'd
 *     memory.  All tensor pointers must be 16-byte aligned.
 *   - bf16 tensors are passed as uint16_t bit patterns, fp16 as uint16_t.
 *   - GQA: query head h reads KV head h / G, G = Hq / Hkv (contiguous groups).
 */
#ifndef VC_H_
#define VC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* vc_stream_t; /* ABI-identical to cudaStream_t */

typedef enum {
  VC_OK = 0,
  VC_ERR_INVALID_ARG = 1, /* NULL / misaligned pointer, negative or inconsistent size */
  VC_ERR_UNSUPPORTED = 2, /* valid but not built: bits not in {2,4,8}, d not in {64,128}, G > 8 ... */
  VC_ERR_CUDA = 3,        /* a CUDA runtime call failed (text in vc_last_error) */
  VC_ERR_TIMEOUT = 4,     /* a bounded wait expired (host event wait or device barrier) */
  VC_ERR_WORKSPACE = 5,   /* workspace pointer NULL or smaller than *_workspace_size() */
  VC_ERR_CAPACITY = 6     /* a length would exceed the capacity the caller allocated */
} vc_status_t;

/* Attention shape shared by the calls below.  Fields a call does not use are
 * ignored (each call lists the ones it reads). */
typedef struct {
  int32_t B;             /* requests in the batch */
  int32_t Hq;            /* query heads */
  int32_t Hkv;           /* KV heads, Hq % Hkv == 0, G = Hq / Hkv <= 8 */
  int32_t d;             /* head dim: 64 or 128 */
  int32_t k;             /* draft length; verify has k + 1 rows per request */
  int32_t bits;          /* KIVI code width: 2, 4 or 8 */
  float softmax_scale;   /* logits = softmax_scale * q . k */
} vc_shape_t;

/* ------------------------------------------------------------ libvc_core */

/* Static text for a status code. */
const char* vc_status_str(vc_status_t s);
/* Reason of the last failing call on this thread ("" if none).  The pointer
 * stays valid until the next failing call on the same thread. */
const char* vc_last_error(void);

/* ------------------------------------------------------- libvc_quant_kv
 * KIVI-style quantiser (VeriCache, Architecture Support: KIVI is one of the
 * quantisation methods the compressor interface takes).  Per group of 32
 * values: s = fp16((max - min) / (2^b - 1)), z = fp16(min),
 * code = clamp(rint((x - z) / s), 0, 2^b - 1) with round-half-even (0 if
 * s == 0); dequantised x^ = fma(code, s, z) in fp32.  Keys group along 32
 * tokens of one channel, values along 32 channels of one token.  The codes
 * are those of this recipe in fp32 with a correctly rounded subtract and
 * divide, bit for bit (the kernel reaches them through a per-group reciprocal
 * and takes the division itself only near a rounding tie).  Inputs are
 * expected finite; a NaN element gets code 0.
 *
 * Packed draft cache of capacity T_cap tokens (T_cap % 32 == 0), NG = T_cap / 32
 * groups of 32 tokens.  The bit placement is this library's own format: it
 * follows the operand fragments of the 16x8x16 fp16 tensor-core product that
 * reads it (two codes an operand register needs sit 16 bits apart in one word).
 *   kc  uint32 [B, Hkv, NG, d*bits]     K codes of a group: 32 lanes x d*bits/32 words,
 *                                       word w of lane L at (w/4)*128 + 4L + w%4
 *   ksz fp16   [B, Hkv, NG, 2, d]       scales of the group's channels, then zeros
 *   vc  uint32 [B, Hkv, NG, d*bits]     V codes, same word order, other field map
 *   vsz fp16   [B, Hkv, NG, d/32, 2, 32]  per channel group: scales, then zeros,
 *                                       entry 8c + 4s + 2r + e = token 8c + 4e + 2s + r
 * Fields (bit 0 = least significant):
 *   bits = 2: slot (u, r, e) starts at 16e + 4u + 2(1 - r);
 *   bits = 4: slot (u, e) starts at 16e + 4u;  bits = 8: at 16e + 8u.
 * Lane L = 4a + c.  K: tokens 4a + j (j < 4), channels (d/4)c + 4k + 2r + e
 * (k < d/16), fragment i = j*(d/16) + k.  V: tokens 8c + 4e + 2s + r, channels
 * 8n + a (n < d/8), fragment i = s*(d/8) + n.  bits = 2: word i/4, u = i%4;
 * bits = 4, 8: i2 = 2i + r, SPW = 16/bits slots per word, word i2/SPW, u = i2%SPW.
 * Bytes per token per KV head: d*bits/4 (codes) + d/4 (metadata).
 */

/* Byte sizes of the four packed arrays for B, Hkv, d, bits and T_cap. */
vc_status_t vc_quant_packed_bytes(const vc_shape_t* s, int32_t T_cap, size_t* kc_bytes,
                                  size_t* ksz_bytes, size_t* vc_bytes, size_t* vsz_bytes);

/* Quantise and pack the first T tokens (T % 32 == 0, T <= T_cap) of
 * K, V bf16 [B, Hkv, T, d] (device, contiguous) into groups 0 .. T/32 - 1 of
 * the packed cache (device).  Reads B, Hkv, d, bits. */
vc_status_t vc_quant_kv_pack(const vc_shape_t* s, int32_t T, int32_t T_cap, const uint16_t* K,
                             const uint16_t* V, uint32_t* kc, uint16_t* ksz, uint32_t* vc,
                             uint16_t* vsz, vc_stream_t stream);

/* Dequantise groups 0 .. T/32 - 1 of a packed cache into fp32
 * K_hat, V_hat [B, Hkv, T, d] (device).  For tests and inspection. */
vc_status_t vc_quant_kv_unpack(const vc_shape_t* s, int32_t T, int32_t T_cap, const uint32_t* kc,
                               const uint16_t* ksz, const uint32_t* vc, const uint16_t* vsz,
                               float* K_hat, float* V_hat, vc_stream_t stream);

/* Commit the accepted tokens to the draft cache and pack full groups
 * (VeriCache, Core Algorithm: the loop repeats from the last accepted token).
 * For every request b (device arrays):
 *   1. append the exact K/V of the n_acc[b] + 1 committed verify inputs,
 *      k_new/v_new bf16 [B, k+1, Hkv, d] rows 0 .. n_acc[b], to the bf16
 *      tail [B, Hkv, tail_cap, d] at tail_len[b] (draft-time entries past
 *      tail_len[b] are overwritten: they are dropped);
 *   2. while the tail holds >= 32 tokens, quantise its oldest 32 into group
 *      packed_len[b] / 32 of the packed cache, packed_len[b] += 32, and shift
 *      the tail down by 32.
 * tail_len and packed_len (int32 [B], device) are updated in place.  If a
 * request would overflow tail_cap or T_cap, it is left unchanged and the
 * device status flag is raised (vc_quant_kv_device_status).
 * n_acc may be NULL to append all k + 1 rows.  Reads B, Hkv, d, k, bits. */
vc_status_t vc_quant_kv_append(const vc_shape_t* s, const uint16_t* k_new, const uint16_t* v_new,
                               const int32_t* n_acc, uint16_t* tail_k, uint16_t* tail_v,
                               int32_t* tail_len, int32_t tail_cap, uint32_t* kc, uint16_t* ksz,
                               uint32_t* vc, uint16_t* vsz, int32_t* packed_len, int32_t T_cap,
                               vc_stream_t stream);

/* SnapKV-style token score (VeriCache, Architecture Support: SnapKV is one
 * of the token-dropping methods the interface takes).  For each request b
 * and KV head: score[t] = sum over the G query heads of the group and over
 * the n_obs observation queries i of softmax_i(t), where query i sits at
 * position T - n_obs + i and sees keys 0 .. T - n_obs + i.
 * q_obs bf16 [B, Hq, n_obs, d], K bf16 [B, Hkv, T, d] -> score fp32
 * [B, Hkv, T] (all device; q_obs and K 16-byte aligned, VC_ERR_INVALID_ARG
 * otherwise).  Logits on the tcgen05 tensor cores (bf16 products, exact,
 * summed in fp32 in TMEM; softmax scale applied in fp32), softmax weights and
 * their sums in fp32.  n_obs <= 32, G * n_obs in 16 * {1, 2, 4, 6, .., 16},
 * T >= n_obs.  Workspace: per (b, KV head) the (max, sum) of every
 * 1024-token range and one threshold M + log2 S per row.  A driver without
 * cuTensorMapEncodeTiled gives VC_ERR_CUDA.
 * Reads B, Hq, Hkv, d, softmax_scale. */
vc_status_t vc_token_score_workspace_size(const vc_shape_t* s, int32_t T, int32_t n_obs,
                                          size_t* bytes);
vc_status_t vc_token_score(const vc_shape_t* s, int32_t T, int32_t n_obs, const uint16_t* q_obs,
                           const uint16_t* K, float* score, void* workspace,
                           size_t workspace_bytes, vc_stream_t stream);

/* Token selection: pooled[t] = max(score[t - pool/2 .. t + pool/2]) (window
 * clipped at the ends); keep the last keep_last tokens and the
 * keep - keep_last tokens of 0 .. T - keep_last - 1 with the largest pooled
 * score (ties -> lower index).  idx int32 [B, Hkv, keep] ascending (device).
 * pool odd, 1 <= pool <= 15; keep_last <= keep <= T. */
vc_status_t vc_token_select_workspace_size(int32_t B, int32_t Hkv, int32_t T, size_t* bytes);
vc_status_t vc_token_select(int32_t B, int32_t Hkv, int32_t T, const float* score, int32_t keep,
                            int32_t keep_last, int32_t pool, int32_t* idx, void* workspace,
                            size_t workspace_bytes, vc_stream_t stream);

/* Gather kept tokens: out[b, h, j] = X[b, h, idx[b, h, j]] for K and V,
 * bf16 [B, Hkv, T, d] -> [B, Hkv, keep, d] (device).  Indices must lie in
 * [0, T); an out-of-range index raises the device status flag and writes
 * zeros.  Reads B, Hkv, d. */
vc_status_t vc_gather_kv(const vc_shape_t* s, int32_t T, int32_t keep, const int32_t* idx,
                         const uint16_t* K, const uint16_t* V, uint16_t* K_out, uint16_t* V_out,
                         vc_stream_t stream);

/* Staging of a packed cache from pinned host memory (VeriCache, Architecture
 * Support, Remote Prefix Caching: the compressed KV is what travels over the
 * slow link to the GPU that drafts).  Copies groups [g0, g1) of every
 * (request, KV head) from host arrays laid out like the device arrays but with
 * host_ng groups per (b, h) (kc, vc: d*bits words per group; ksz, vsz: 2*d
 * fp16 per group) into the device arrays of capacity T_cap: four 2-D
 * host-to-device copies on `stream`, no kernel.  The host arrays must be
 * pinned (checked) and stay untouched until the copies complete.  Sets no
 * lengths: the caller sets packed_len once the groups it needs have landed.
 * Reads B, Hkv, d, bits. */
vc_status_t vc_quant_kv_stage_groups(const vc_shape_t* s, const uint32_t* host_kc, const uint16_t* host_ksz,
                                     const uint32_t* host_vc, const uint16_t* host_vsz, int32_t host_ng,
                                     int32_t g0, int32_t g1, int32_t T_cap, uint32_t* kc, uint16_t* ksz,
                                     uint32_t* vc, uint16_t* vsz, vc_stream_t stream);

/* Device status of libvc_quant_kv kernels since the last call: 0 = none.
 * Synchronises the device; clears the flag. */
vc_status_t vc_quant_kv_device_status(uint32_t* status);

/* ------------------------------------------------------ libvc_draft_attn
 * Draft decode attention over the compressed cache (VeriCache, Core
 * Algorithm, Drafting; Key System Innovations: drafting is bound by HBM
 * bandwidth).  For request b and query head h:
 *   o = softmax(scale * q . [K^ ; tail_k[0 : tail_len[b] + step] ; k_cur]^T)
 *       [V^ ; tail_v[...] ; v_cur]
 * with K^, V^ the dequantised packed tokens 0 .. packed_len[b] - 1.
 * If k_cur/v_cur (bf16 [B, Hkv, d]) are given, they are also stored at tail
 * position tail_len[b] + step (for the following draft steps); if NULL, the
 * current token is not added and the tail is not written.
 * q bf16 [B, Hq, d] -> out bf16 [B, Hq, d].  packed_len, tail_len: int32 [B]
 * device.  max_packed: an upper bound of packed_len over the batch (host);
 * the launch's partition spreads max_packed / 32 groups a slice over the
 * SMs, so the tightest bound balances best.
 * One launch: the packed groups of all (request, KV head) slices are split
 * evenly over a persistent grid sized to the current device (stream-K), the
 * partials are merged with a log-sum-exp rule by the last CTA of each slice.
 * The packed tokens go through fp16 tensor-core products with fp32
 * accumulation: each code field, masked in place, is the fp16 subnormal
 * code * 2^(p - 24); key scales (and the fields' powers of two) fold into the
 * query and value scales into the softmax weights, as single fp16 values.
 * Range limits of those fp16 operands (every code width): |q| * key scale * 16
 * and 8 * 16 * value scale must stay below 65504.
 * G = Hq / Hkv in {1, 2, 4, 5, 8}; softmax_scale > 0.
 * The workspace holds the partials and one arrival
 * counter per slice: it must be zero-filled before its first use, and every
 * call leaves the counters at zero again.  Its size depends on the device
 * (SM count, occupancy) and the shape: query it with the same device
 * current.  A size queried with some max_packed > 0 serves calls of the same
 * shape with every max_packed.  Calls that
 * share a workspace must not overlap on the GPU, other than as chained calls
 * (below), which order their workspace accesses themselves.
 * flags: 0, or VC_DRAFT_CHAINED for a call enqueued directly after another
 * vc_draft_attn call on the same stream, with no other work between them
 * (the draft steps of a round, layer after layer).  Such a call is launched
 * with programmatic dependent launch: its CTAs may start while the previous
 * call's last CTAs run, and before that call has finished they read only
 * this call's packed cache (kc, ksz, vc, vsz, packed_len), which no draft
 * call writes; queries, k_cur/v_cur, the tail, the workspace and out are
 * touched only after it.  So work that writes a packed cache (pack, append,
 * staging) goes before a chain's first, unchained call.  Other bits:
 * VC_ERR_INVALID_ARG.
 * Reads B, Hq, Hkv, d, bits, softmax_scale. */
#define VC_DRAFT_CHAINED 1u
vc_status_t vc_draft_attn_workspace_size(const vc_shape_t* s, int32_t max_packed, size_t* bytes);
vc_status_t vc_draft_attn(const vc_shape_t* s, const uint16_t* q, const uint16_t* k_cur,
                          const uint16_t* v_cur, const uint32_t* kc, const uint16_t* ksz,
                          const uint32_t* vc, const uint16_t* vsz, const int32_t* packed_len,
                          int32_t max_packed, int32_t T_cap, uint16_t* tail_k, uint16_t* tail_v,
                          const int32_t* tail_len, int32_t tail_cap, int32_t step, uint16_t* out,
                          void* workspace, size_t workspace_bytes, uint32_t flags, vc_stream_t stream);
/* Device status (barrier time-outs) since the last call; synchronises. */
vc_status_t vc_draft_attn_device_status(uint32_t* status);
/* The stream-K partition a vc_draft_attn launch uses, computed on the host
 * (no device access), for inspection and tests.  The packed groups of the
 * B * Hkv slices (max_packed / 32 each) are laid end to end, slice-major.
 * slots is the launch's CTA slots: occupancy x SM count, one CTA per SM for
 * this kernel.  Outputs:
 *   n_stream   the stream CTAs: at most slots (and 512), at most one per 11
 *              groups, 0 when max_packed is 0;
 *   lo         lo[0 .. n_stream]: CTA c takes groups [lo[c], lo[c + 1]);
 *              lo[0] = 0 and lo[n_stream] = the groups in all;
 *   max_parts  partial slots of a slice: the bound of stream CTAs that meet
 *              one slice, plus the tail's slot.
 * A CTA's range is balanced by cost: its groups, plus a charge per slice
 * boundary inside it and per bf16 tail pass it runs, scaled by the bytes of
 * a group.  lo_len < n_stream + 1: VC_ERR_INVALID_ARG. */
vc_status_t vc_draft_attn_partition(const vc_shape_t* s, int32_t max_packed, int32_t slots, int32_t* n_stream,
                                    int32_t* lo, int32_t lo_len, int32_t* max_parts);
/* Test hooks, for the failure-detection test only (host-side settings of this
 * library, not thread-safe, apply to later vc_draft_attn calls):
 *   wait_cycles           bound of every mbarrier wait of the draft kernel in
 *                         SM clock cycles; 0 restores the default (about 2 s),
 *                         otherwise >= 1000;
 *   withhold_first_stage  1: each stream CTA's producer issues no copy for its
 *                         first ring stage, so that stage's consumers' waits
 *                         run out; 0: normal.
 * A call that ran out raises the barrier time-out bit of
 * vc_draft_attn_device_status, leaves its output undefined and its workspace
 * dirty: zero the workspace before reusing it.  No wait is unbounded and no
 * fault is raised.  With a short bound, do not chain calls
 * (VC_DRAFT_CHAINED): a chained call's producer fills its ring and then waits
 * for consumers that themselves wait for the previous call, and that wait
 * counts against the bound. */
vc_status_t vc_draft_attn_test_hooks(int64_t wait_cycles, int32_t withhold_first_stage);

/* ----------------------------------------------------- libvc_verify_attn
 * Verify attention (VeriCache, Core Algorithm, Verification: one forward
 * pass over the full KV checks all drafted tokens at once).  Verify row j in
 * 0 .. k (inputs [t_last, d_0 .. d_{k-1}]) of request b, query head h:
 *   o = softmax(scale * q_j . [K[0 : prefix_len[b]] ; k_new[0 .. j]]^T) [V ; v_new]
 * The full KV lives in pinned host memory (Architecture Support) in chunks
 * of C tokens, chunk-major:
 *   host_kv bf16 [n_chunks_cap][2 (K, V)][B][Hkv][C][d]
 * so that one chunk is one contiguous host->device copy into a device slot
 * bf16 [2][B][Hkv][C][d].
 * q bf16 [B, k+1, Hq, d]; k_new, v_new bf16 [B, k+1, Hkv, d]; out bf16
 * [B, k+1, Hq, d].  Rows per KV head M = (k+1) * G <= 512.  Tensor-core
 * (bf16 MMA, fp32 accumulate) QK^T and PV; split-KV partials merged with a
 * log-sum-exp rule.  Reads B, Hq, Hkv, d, k, softmax_scale.
 *
 * Workspace: parts_per_chunk running partial states + one for the new tokens.
 */
vc_status_t vc_verify_attn_workspace_size(const vc_shape_t* s, int32_t parts_per_chunk, size_t* bytes);

/* Parts per chunk (split-KV partitions of one chunk launch) for this shape
 * and chunk length C on the current device: chosen from the chunk kernel's
 * occupancy so the launch's CTAs fill the SMs in whole waves, with the fewest
 * tiles per CTA (1 <= parts <= 16).  Pass the result as parts_per_chunk.
 * Host-only: queries the device, launches nothing. */
vc_status_t vc_verify_attn_parts(const vc_shape_t* s, int32_t C, int32_t* parts);

/* Low-level, one chunk already in device memory: merge its tokens
 * [chunk_start, chunk_start + C) of every request (only those below
 * prefix_len[b]) into the running partial state.  first != 0 starts a new
 * pass (overwrites the state). */
vc_status_t vc_verify_attn_chunk(const vc_shape_t* s, const uint16_t* q, const uint16_t* kv_slot,
                                 int32_t C, int32_t chunk_start, const int32_t* prefix_len,
                                 int32_t parts_per_chunk, int32_t first, void* workspace,
                                 size_t workspace_bytes, vc_stream_t stream);
/* The causal block of the k + 1 new tokens, then the final combine -> out. */
vc_status_t vc_verify_attn_finish(const vc_shape_t* s, const uint16_t* q, const uint16_t* k_new,
                                  const uint16_t* v_new, int32_t parts_per_chunk,
                                  int32_t any_chunk, uint16_t* out, void* workspace,
                                  size_t workspace_bytes, vc_stream_t stream);

/* Streamed pipeline: events for a ring of n_slots device slots. */
typedef struct vc_verify_pipeline* vc_verify_pipeline_t;
vc_status_t vc_verify_pipeline_create(int32_t n_slots, vc_verify_pipeline_t* p);
vc_status_t vc_verify_pipeline_destroy(vc_verify_pipeline_t p);

/* Host-side prefetch of chunks [0, n_chunks) on the copy stream into ring
 * slots, as far as free slots allow, without the compute side.  Lets a
 * caller start the transfer before the verify queries exist (e.g. while
 * drafting).  Tokens at or beyond max_prefix are not copied.  T_cap is the
 * pinned store's capacity in tokens per request (a multiple of C, the same
 * value vc_verify_commit takes); max_prefix > T_cap is an argument error, so
 * no copy reads past the store. */
vc_status_t vc_verify_prefetch(vc_verify_pipeline_t p, const vc_shape_t* s,
                               const uint16_t* host_kv, int32_t C, int32_t max_prefix,
                               int32_t T_cap, uint16_t* dev_slots, vc_stream_t copy_stream);

/* Whole verify for one layer: streams chunks 0 .. ceil(max_prefix / C) - 1
 * of host_kv (pinned, T_cap / C chunks) through the ring dev_slots (device,
 * n_slots slots of 2*B*Hkv*C*d bf16 each) on copy_stream, runs the chunk
 * kernels on compute_stream as chunks land (CUDA events, no host waits), then
 * the new tokens and the combine.  max_prefix (host) bounds prefix_len[b]
 * (device) and must not exceed T_cap. */
vc_status_t vc_verify_attn_streamed(vc_verify_pipeline_t p, const vc_shape_t* s,
                                    const uint16_t* q, const uint16_t* host_kv, int32_t C,
                                    int32_t max_prefix, int32_t T_cap, const int32_t* prefix_len,
                                    uint16_t* dev_slots, const uint16_t* k_new,
                                    const uint16_t* v_new, uint16_t* out, int32_t parts_per_chunk,
                                    void* workspace, size_t workspace_bytes,
                                    vc_stream_t compute_stream, vc_stream_t copy_stream);

/* Commit the exact K/V of the n_acc[b] + 1 accepted verify inputs (rows
 * 0 .. n_acc[b] of k_new/v_new) into the pinned host store at token
 * prefix_len[b] and advance prefix_len[b] (device, in place).  The kernel
 * writes host memory directly (mapped pinned memory).  A request that would
 * pass T_cap (= n_chunks_cap * C) is left unchanged and raises the device
 * status flag.  n_acc may be NULL (commit all k + 1 rows). */
vc_status_t vc_verify_commit(const vc_shape_t* s, const uint16_t* k_new, const uint16_t* v_new,
                             const int32_t* n_acc, int32_t* prefix_len, uint16_t* host_kv,
                             int32_t C, int32_t T_cap, vc_stream_t stream);

/* Device status of libvc_verify_attn kernels since the last call; synchronises. */
vc_status_t vc_verify_attn_device_status(uint32_t* status);

/* ------------------------------------------------------------ libvc_accept
 * Acceptance (VeriCache, Core Algorithm, Acceptance).  For request b:
 * a_i = argmax_v logits[b, i, v] (ties -> lowest v, IEEE comparisons) for
 * i in 0 .. k; n_acc[b] = first i < k with a_i != draft[b, i], else k;
 * next_tok[b] = a_{n_acc[b]} (the bonus token when n_acc == k, the full-KV
 * correction otherwise).  logits fp32 [B, k+1, V], draft int32 [B, k];
 * outputs int32 (device); argmax int32 [B, k+1] optional (NULL to skip).
 * NaN logits are unsupported.  The workspace starts with B per-request
 * arrival counters at a fixed place: zero-fill the workspace before its first
 * use; every call leaves the counters at zero, so one workspace, sized for the
 * largest need, serves calls with any k and V for the same B (the size is not
 * monotone in k: query it for every k that will be used). */
vc_status_t vc_accept_workspace_size(int32_t B, int32_t k, int32_t V, size_t* bytes);
vc_status_t vc_accept(int32_t B, int32_t k, int32_t V, const float* logits, const int32_t* draft,
                      int32_t* n_acc, int32_t* next_tok, int32_t* argmax, void* workspace,
                      size_t workspace_bytes, vc_stream_t stream);

/* vc_accept without a workspace argument and without any allocation.  The
 * paper has no counterpart: this exists for callers that cannot allocate
 * device memory, such as a plugin that a serving framework gives only its
 * input and output buffers (the framework owns all device memory), or a
 * latency-critical loop where cudaMalloc, which may synchronise the device,
 * is not allowed.  Same inputs, outputs and results as vc_accept.
 *
 * Scratch lives in a fixed 64 KiB array in the library's device memory, which
 * every GPU that loads libvc_accept.so holds until the process exits.  Limits:
 * B <= 4096 and B*(k+1)*S <= 6144, S = splits per row = min(ceil(1216 /
 * (B*(k+1))), ceil(V / 2048)), at least 1 (e.g. B=8, k=16, V=32768 uses
 * 1224); larger calls return VC_ERR_CAPACITY with the reason.  Every call
 * looks up the array's address on the current device (cudaGetSymbolAddress,
 * a host query that allocates nothing), so a context made after a
 * cudaDeviceReset gets its own.  The first call on a device also loads the
 * library's module there: make it before any stream capture.  Each call
 * zeroes the counters it needs on the stream before its kernel.  All calls
 * share the one array: calls that overlap on the GPU (other streams, other
 * host threads) race and return wrong results.  No cudaMalloc / cudaFree or
 * allocating library routine is called. */
vc_status_t vc_accept_noalloc(int32_t B, int32_t k, int32_t V, const float* logits,
                              const int32_t* draft, int32_t* n_acc, int32_t* next_tok,
                              int32_t* argmax, vc_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* VC_H_ */
