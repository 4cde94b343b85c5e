/*
 * attn.h -- C ABI of libattn.so: fused softmax attention forward on one GB300.
 *
 * Every entry point computes, for each batch entry b, query head h and query
 * row i,
 *
 *     O[b,h,i,:] = softmax_k( scale * Q[b,h,i,:] . K[b,g,k,:] + mask[b,h,i,k] ) V[b,g,k,:]
 *     LSE[b,h,i] = log sum_k exp( scale * Q . K + mask )          (natural log)
 *
 * with g = h / (heads / kv_heads), the sum running over the keys visible to the
 * row.  Sources: "Attention" (recursiveai.org OneGPU docs), opening paragraph
 * (the formula and the online normaliser), section "What it covers" (element
 * types, layouts, lengths, heads, head dimension, masks) and section "Special
 * values"; "attention_forward -- Causal Multi-Head Attention with Online
 * Softmax" (llm.istanbul), sections "GQA", "2) Phase 0" (segment starts) and
 * "Online Softmax Algoritmasi" (LSE = m + log l); "com.microsoft.GroupQueryAttention"
 * (webgpu-kernels README), section "Inputs" (BNSH key/value caches, per-sample
 * key lengths, additive attention bias with broadcast leading dimensions).
 *
 * Key visibility.  Key k (0 <= k < k_len) is visible to row (b, i) iff
 *   - k < L_b = clamp(k_lens[b], 0, k_len)    when k_lens is given (L_b = k_len otherwise;
 *                                             k_lens[b] + 1 under ATTN_KLENS_LAST_INDEX), and
 *   - k <= i + off_b                          when causal != 0, with off_b = causal_offset,
 *                                             or L_b - q_len under ATTN_CAUSAL_KLENS, and
 *   - k >= i + off_b - window_left            when causal != 0 and window_left >= 0, and
 *   - k >= clamp(seg[b, i], 0, k_len)         when seg is given,
 * and its weight is zero when mask[b,h,i,k] = -inf.  A visible key whose score
 * is NaN or +inf makes the whole row NaN (O and LSE).  A row with no key of
 * non-zero weight (k_len = 0 included) gives NaN in every O element, or 0
 * under ATTN_MASKED_ROWS_ZERO, and LSE = -inf.  Out-of-range k_lens and seg
 * values are clamped to [0, k_len] (a convention of this library).
 *
 * Score transforms ("com.microsoft.GroupQueryAttention", attributes softcap
 * and smooth_softmax, input head_sink).  With softcap c > 0 the scaled dot
 * product s becomes c * tanh(s / c) before the mask is added.  With a sink,
 * the logit sigma_h (head_sink[h], or 0 under smooth_softmax alone) joins
 * every row's denominator as exp(sigma_h) and adds nothing to the numerator;
 * LSE is the log of the whole denominator.  A row with a sink and no visible
 * key gives O = 0 and LSE = sigma_h; a NaN or +inf sink makes the row NaN; a
 * sink of -inf adds nothing.
 *
 * Quantised key/value cache ("com.microsoft.GroupQueryAttention", inputs
 * k_scale and v_scale, attributes k_quant_type, v_quant_type and
 * kv_cache_bit_width = 8).  With kv_dtype = ATTN_KV_INT8 the K and V elements
 * are signed 8-bit integers (layouts in elements = bytes) and an element's
 * value is the integer times its float32 scale: k_scale[0] for every element
 * (ATTN_KV_SCALE_TENSOR) or k_scale[g * head_dim + d] for kv head g, channel d
 * (ATTN_KV_SCALE_CHANNEL); likewise v_scale.  Q and O keep dtype.
 *
 * Memory.  Every data pointer is a DEVICE pointer owned by the caller.  The
 * library allocates no device memory: scratch space is the caller's
 * `workspace` (size from the *_workspace_size queries).  K/V values of keys
 * that are hidden from every query row of a 128-row query tile are never read
 * into the result; V values of a key that some row of the tile sees must be
 * finite, or rows of that tile that hide the key may become NaN (tensor-core
 * products multiply them by zero).
 *
 * Execution.  Calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 * legacy default stream): they validate on the host, enqueue kernels and
 * return.  No call synchronises the host except attn_device_status.  No C++
 * exception crosses the ABI.  Results are deterministic: every sum has a
 * fixed order and no float atomics are used, so two runs give identical bits.
 * Calls on one stream are serialised by the stream; concurrent calls on
 * different streams must not share output or workspace buffers.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* attn_stream;

/* Element type of Q, K, V and O.  The mask and LSE are always float32. */
enum { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 };

/* What a row with no visible key returns ("Attention", section "Special values"). */
enum { ATTN_MASKED_ROWS_NAN = 0, ATTN_MASKED_ROWS_ZERO = 1 };

/* Status codes. */
enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* null required pointer, negative size, heads % kv_heads != 0,
                                  head_dim outside [1, 256], odd head_dim for f16/bf16, bad layout,
                                  window_left < -1 or a window without causal, unknown enum value,
                                  negative or non-finite softcap, int8 K/V without scales */
  ATTN_ERR_UNSUPPORTED = 2,    /* a valid combination this build does not implement */
  ATTN_ERR_ALIGNMENT = 3,      /* a pointer not aligned to its element size */
  ATTN_ERR_WORKSPACE = 4,      /* workspace missing or smaller than the size query says */
  ATTN_ERR_CUDA = 5,           /* a CUDA runtime/driver call or a launch failed */
  ATTN_ERR_DEVICE_TIMEOUT = 6  /* a kernel gave up a bounded wait (see attn_device_status) */
};

/* ATTN_OFFSET_DEFAULT as causal_offset selects k_len - q_len ("Attention",
 * section "What it covers": the cached-decoder default). */
#define ATTN_OFFSET_DEFAULT INT64_MIN

/* Where the causal diagonal sits ("com.microsoft.GroupQueryAttention",
 * chunked-prefill variants: the causal bound of each sample is right-aligned
 * to its live length).  ATTN_CAUSAL_FIXED: one offset for every batch entry
 * (causal_offset).  ATTN_CAUSAL_KLENS: batch entry b's offset is L_b - q_len,
 * so its last query row sees exactly its L_b valid keys. */
enum { ATTN_CAUSAL_FIXED = 0, ATTN_CAUSAL_KLENS = 1 };

/* Meaning of k_lens[b] ("com.microsoft.GroupQueryAttention", input seqlens_k):
 * ATTN_KLENS_COUNT: the number of valid keys; ATTN_KLENS_LAST_INDEX: the index
 * of the last valid key, i.e. the count minus one (ONNX seqlens_k as given). */
enum { ATTN_KLENS_COUNT = 0, ATTN_KLENS_LAST_INDEX = 1 };

/* Storage of K and V (see "Quantised key/value cache" above). */
enum { ATTN_KV_AS_Q = 0, ATTN_KV_INT8 = 1 };
enum { ATTN_KV_SCALE_TENSOR = 0, ATTN_KV_SCALE_CHANNEL = 1 };

/* A strided 4-D view [batch][head][row][element]: element (b, h, r, e) is at
 * base[offset + b*batch_stride + h*head_stride + r*row_stride + e].  Strides
 * are in elements; the elements of a row are contiguous.  Position-first
 * [B, S, H, D] is {0, S*H*D, D, H*D}; head-first [B, H, S, D] is
 * {0, H*S*D, S*D, D}; a slice of a packed QKV projection sets offset. */
typedef struct {
  int64_t offset, batch_stride, head_stride, row_stride;
} attn_layout;

/* The problem ("Attention", section "What it covers"; P(batch, heads, qLen,
 * kLen, headDim) of that page's example, plus kv_heads for grouped heads). */
typedef struct {
  int32_t batch, heads, kv_heads;  /* heads % kv_heads == 0 */
  int32_t q_len, k_len;            /* k_len is the cache capacity for attn_decode */
  int32_t head_dim;                /* 1..256; even for f16/bf16 */
  int32_t dtype;                   /* ATTN_F32 / ATTN_F16 / ATTN_BF16 */
  float scale;                     /* 0 selects the float nearest 1/sqrt(head_dim) */
  int32_t causal;                  /* 0 or 1 */
  int64_t causal_offset;           /* used iff causal; ATTN_OFFSET_DEFAULT = k_len - q_len */
  int32_t masked_rows;             /* ATTN_MASKED_ROWS_NAN / ATTN_MASKED_ROWS_ZERO */
  attn_layout q, k, v, o;          /* Q, O over heads; K, V over kv_heads */
  attn_layout mask;                /* float32 mask strides over (batch, head, row); 0 broadcasts;
                                      keys contiguous.  Ignored when mask == NULL. */
  int64_t seg_batch_stride;        /* seg is int32 [batch][q_len] with this batch stride (0 shares one row set) */
  int64_t lse_batch_stride;        /* LSE float32 element (b, h, i) at lse[b*lse_batch_stride + */
  int64_t lse_head_stride;         /*   h*lse_head_stride + i] */
  /* Visibility variants ("com.microsoft.GroupQueryAttention", attribute
   * local_window_size, input seqlens_k, chunked-prefill causal bound). */
  int32_t window_left;             /* -1: off.  With causal, row i keeps keys i + off_b - window_left
                                      .. i + off_b (window_left + 1 keys at most).  Requires causal. */
  int32_t causal_align;            /* ATTN_CAUSAL_FIXED / ATTN_CAUSAL_KLENS */
  int32_t k_lens_kind;             /* ATTN_KLENS_COUNT / ATTN_KLENS_LAST_INDEX */
  /* Score transforms (see above). */
  float softcap;                   /* 0: off; > 0: cap of the scaled dot products (finite) */
  int32_t smooth_softmax;          /* 1: the sink term is on, sigma_h = 0 unless head_sink is given */
  const float* head_sink;          /* nullable DEVICE pointer, float32 [heads]: per-head sink logits;
                                      non-NULL turns the sink term on.  Owned by the caller. */
  /* Key/value storage (see above). */
  int32_t kv_dtype;                /* ATTN_KV_AS_Q / ATTN_KV_INT8 */
  int32_t kv_scale_kind;           /* ATTN_KV_SCALE_TENSOR / ATTN_KV_SCALE_CHANNEL */
  const float* k_scale;            /* DEVICE float32 scales, required with ATTN_KV_INT8 */
  const float* v_scale;
  /* Key-range split of attn_fwd ("Attention", section "Accuracy at long key
   * lengths": the keys are cut into ranges by the shape, each range gives a
   * partial (LSE, O), and the partials are merged in range order).  0: the
   * library's plan (ranges only when the problem has too few query blocks to
   * fill the GPU and at least 2048 keys, see attn_fwd_workspace_size);
   * n >= 1: exactly min(n, 16) ranges of equal length (a multiple of 128
   * keys), the last one shorter.  attn_decode ignores it. */
  int32_t key_splits;
} attn_problem;

/* Bytes of device workspace attn_fwd needs for this problem (0 when none):
 * the partial results of its key ranges (float32 [B*H*q_len][ranges][head_dim]
 * and [B*H*q_len][ranges], each 256-byte aligned).  The plan depends on the
 * shape only: without key_splits the keys are cut into ranges when the
 * problem has fewer than 304 blocks of query rows (256 rows a block for
 * head_dim <= 128, 128 above; two blocks per SM of a GB300) and at least
 * 2048 keys: ceil(304 / blocks) ranges, at most 16 and at most one per 1024
 * keys.  Returns 0 also for an invalid problem; attn_fwd then reports the
 * error. */
ATTN_API size_t attn_fwd_workspace_size(const attn_problem* p);

/* Prefill / full forward.  q, k, v, o: device pointers in p->dtype laid out
 * by p->q, p->k, p->v, p->o.  mask (nullable): float32, strides p->mask.
 * seg (nullable): int32 segment starts.  k_lens (nullable): int32 [batch]
 * key counts.  lse (nullable): float32 output.  workspace: device scratch of
 * attn_fwd_workspace_size(p) bytes, 256-byte aligned.  When the plan cuts the
 * keys into ranges, a pass writes each range's partial into the workspace and
 * a second kernel merges them in range order; with a smaller workspace (NULL
 * included) the call runs without ranges, unless p->key_splits > 1 asks for
 * them, which returns ATTN_ERR_WORKSPACE.  The two forms agree within
 * rounding (the sums run in another order); each is deterministic.
 * batch == 0 or q_len == 0 is a no-op returning ATTN_OK. */
ATTN_API int attn_fwd(const attn_problem* p, const void* q, const void* k, const void* v, void* o,
             const float* mask, const int32_t* seg, const int32_t* k_lens, float* lse,
             void* workspace, size_t workspace_bytes, attn_stream stream);

/* Bytes of device workspace attn_decode needs (per-range partial results). */
ATTN_API size_t attn_decode_workspace_size(const attn_problem* p);

/* Single-query decode against a key/value cache: q_len must be 1.  The keys
 * are cut into ranges whose size depends only on the shape (k_len, batch,
 * kv_heads); each range writes a partial (LSE, O) into the workspace and a
 * second kernel merges them in range order (the split-K decode of
 * "com.microsoft.GroupQueryAttention", section "Implementation variants",
 * and the key-range split of "Attention", section "Accuracy at long key
 * lengths").  k_cache/v_cache are laid out by p->k/p->v (BNSH cache:
 * {0, kv_heads*cap*D, cap*D, D}); k_lens (nullable) holds each sample's
 * number of valid cache rows (an ONNX seqlens_k value plus one).  mask, seg and
 * lse are as for attn_fwd and may be NULL. */
ATTN_API int attn_decode(const attn_problem* p, const void* q, const void* k_cache, const void* v_cache,
                void* o, const float* mask, const int32_t* seg, const int32_t* k_lens, float* lse,
                void* workspace, size_t workspace_bytes, attn_stream stream);

/* attn_decode without a caller workspace, for callers that cannot allocate
 * device memory (code handed only a stream, allocator hooks, loops that must
 * not take allocator locks, plugins of a runtime that owns all device memory).
 * The pages describe no such entry point; it is an addition of this library.
 * Same arguments and results as attn_decode minus the workspace: the partial
 * results live in a fixed device array of attn_decode_noalloc_max_scratch()
 * bytes (32 MiB) that this library holds on every GPU it is loaded on until
 * the process exits.  A problem whose attn_decode_workspace_size exceeds that
 * returns ATTN_ERR_WORKSPACE and launches nothing.  The first call on a device
 * looks up the array's device address (once per device); make it before any
 * stream capture.  No call allocates or frees memory.  All calls share the
 * array: calls whose GPU work overlaps (different streams or host threads)
 * race, so serialise them.  The array keeps the last call's contents; every
 * value a call reads was written by that call. */
ATTN_API int attn_decode_noalloc(const attn_problem* p, const void* q, const void* k_cache,
                                 const void* v_cache, void* o, const float* mask, const int32_t* seg,
                                 const int32_t* k_lens, float* lse, attn_stream stream);

/* Decode step with the cache update fused in ("com.microsoft.GroupQueryAttention":
 * present_key / present_value sharing the past buffer; seqlens_k counts the new
 * token; the int8 decode variant appends quantised rows).  Same as attn_decode,
 * except that the caches are written: for every batch entry b with
 * L_b = clamp(k_lens[b] (+1 under ATTN_KLENS_LAST_INDEX), 0, k_len) >= 1 and
 * every kv head g, cache row L_b - 1 first takes the new rows
 * k_new / v_new[(b * kv_heads + g) * head_dim ..] (device, contiguous
 * [batch][kv_heads][head_dim], in dtype), and then the step attends over rows
 * 0 .. L_b - 1 as attn_decode does.  An int8 cache (kv_dtype = ATTN_KV_INT8)
 * stores x / scale rounded to the nearest integer (ties to even, float32
 * division) and saturated to [-128, 127].  k_lens is required; seg is not
 * taken.  The row is written by the kernels of the step itself (no separate
 * copy kernel); the caches must not be read by other work while the step runs. */
ATTN_API int attn_decode_append(const attn_problem* p, const void* q, const void* k_new, const void* v_new,
                                void* k_cache, void* v_cache, void* o, const float* mask, const int32_t* k_lens,
                                float* lse, void* workspace, size_t workspace_bytes, attn_stream stream);

/* Size in bytes of the fixed scratch array attn_decode_noalloc uses. */
ATTN_API size_t attn_decode_noalloc_max_scratch(void);

/* Merge per-range partial results of `rows` rows ("Attention", section
 * "Accuracy at long key lengths": partials merged in range order).
 * part_o: float32 [rows][n_splits][head_dim], each already divided by its own
 * sum; part_lse: float32 [rows][n_splits] (-inf marks an empty range).  The
 * row result is O = sum_r exp(lse_r) O_r / sum_r exp(lse_r) and
 * LSE = log sum_r exp(lse_r), written to o (out_dtype, row r at
 * o + r*o_row_stride elements) and lse (nullable, float32 [rows]).  A NaN or
 * +inf lse_r makes the row NaN; all ranges empty gives a masked row. */
ATTN_API int attn_combine(int32_t n_splits, int32_t rows, int32_t head_dim, const float* part_o,
                 const float* part_lse, int32_t out_dtype, void* o, int64_t o_row_stride, float* lse,
                 int32_t masked_rows, attn_stream stream);

/* Synchronises `stream`, then reads and clears the library's device status
 * word on the current device: ATTN_OK, or ATTN_ERR_DEVICE_TIMEOUT when a
 * kernel abandoned a bounded wait since the last call (its outputs are then
 * undefined).  Returns ATTN_ERR_CUDA if synchronising fails. */
ATTN_API int attn_device_status(attn_stream stream);

/* Static description of a status code. */
ATTN_API const char* attn_status_string(int status);

/* Measurement utility, not part of the attention path.  The softmax takes one
 * base-2 exponential per visible query-key pair ("Attention", opening
 * paragraph), so the hardware exponential's throughput bounds the prefill
 * beside the tensor cores.  This launches `blocks` CTAs of 256 threads on
 * `stream`; every thread evaluates `iters` x 8 approximate exponentials
 * (ex2.approx, eight independent chains) and each CTA writes one float to
 * sink[blockIdx] (device, float32 [blocks], 4-byte aligned, caller-owned) so
 * the work is kept.  The caller times the launch with events: the rate is
 * blocks * 256 * iters * 8 / time.  Returns ATTN_ERR_INVALID_ARG for
 * blocks < 1, iters < 1 or a null or misaligned sink; ATTN_ERR_CUDA if the
 * launch fails. */
ATTN_API int attn_probe_ex2(int32_t blocks, int32_t iters, float* sink, attn_stream stream);

/* Test utility, not part of the attention path: arms a one-shot fault for the
 * tests of the kernels' bounded waits.  With ATTN_INJECT_DROP_FIRST_COPY, the
 * next launch of a tensor-core kernel (the prefill kernels and the decode
 * split passes; the CUDA-core kernels ignore it and leave it armed) makes its
 * first CTA announce its first key-tile copy to the copy's barrier without
 * issuing it.  The waits on that barrier then run out after about 2 s; the CTA
 * records ATTN_ERR_DEVICE_TIMEOUT in the status word (attn_device_status),
 * waits (bounded) for the copies and tensor-core work it did start, frees its
 * tensor memory and exits, so the context stays usable.  That call's outputs
 * are undefined; later calls are unaffected.  ATTN_INJECT_NONE disarms.
 * The fault is process-wide and host-side: nothing outside this call arms it.
 * Returns ATTN_ERR_INVALID_ARG for an unknown code. */
enum { ATTN_INJECT_NONE = 0, ATTN_INJECT_DROP_FIRST_COPY = 1 };
ATTN_API int attn_test_inject(int32_t fault);

/* Library version as major*10000 + minor*100 + patch. */
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
