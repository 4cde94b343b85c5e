/*
 * attn_oracle.c -- float64 CPU oracle for fused softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load or run this library.  It shares no
 * code, header, table or helper with the CUDA path, and it never reads
 * anything the CUDA path produced.
 *
 * What it computes is the plain definition of the method, not the method's
 * fast algorithm:
 *
 *   O = softmax(Scale * Q K^T + Mask) V, per batch entry and head
 *     -- "Attention" (recursiveai.org OneGPU docs), opening paragraph.
 *
 * written as the classic three-pass softmax per query row (row max, then the
 * sum of exp(s - max), then the normalised weighted sum of V) -- "attention_forward
 * -- Causal Multi-Head Attention with Online Softmax" (llm.istanbul), section
 * "Online Softmax -- Niye?".  The online normaliser of the GPU kernels is an
 * exact rearrangement of this, so the definition is the oracle.
 *
 * Key visibility, special values and element types follow "Attention",
 * sections "What it covers" and "Special values"; the grouped-head mapping
 * kv_h = h / (heads / kv_heads) follows "attention_forward ...", section "GQA";
 * the segment rule (keys before the row's document start are hidden) follows
 * "attention_forward ...", section "2) Phase 0"; LSE = m + log(l) follows the
 * "final:" step of that page's "Online Softmax Algoritmasi" section.
 *
 * Readings where the pages are silent (all mirrored by the CUDA path as a
 * documented convention, not by shared code):
 *   - device key lengths and segment starts are clamped to [0, k_len];
 *   - a row with no visible key has LSE = -inf (the log of an empty sum);
 *   - a row with a NaN or +inf score among its visible keys gives NaN in
 *     every output element and NaN LSE, in both masked-rows modes;
 *   - the default causal offset is k_len - q_len; the default scale is the
 *     float32 value nearest 1/sqrt(head_dim);
 *   - local (sliding-window) attention with left window w keeps, for a causal
 *     row whose diagonal key is i + offset, the keys i + offset - w .. i +
 *     offset (w + 1 keys at most; w = 0 keeps the diagonal key alone);
 *   - the right-aligned causal bound of chunked prefill uses, for batch entry
 *     b, the offset (clamped key length of b) - q_len in place of the single
 *     offset;
 *   - key lengths given as "last index" (ONNX seqlens_k) are counts minus one.
 *
 * The three visibility variants follow "com.microsoft.GroupQueryAttention"
 * (webgpu-kernels README): attribute local_window_size, input seqlens_k, and
 * its chunked-prefill variants, whose causal bound is right-aligned to each
 * sample's live length.
 *
 * Score transforms, from the same page (attributes softcap and
 * smooth_softmax, input head_sink), with these readings:
 *   - soft-capping with cap c > 0 replaces the scaled dot product s by
 *     c * tanh(s / c); the additive mask is added after it (so a -inf mask
 *     still hides its key);
 *   - the per-head sink value sigma_h is a logit that joins every row's
 *     softmax denominator as exp(sigma_h) and adds nothing to the numerator;
 *     smooth_softmax without per-head values uses sigma_h = 0 (the "+1" of the
 *     smooth-softmax denominator).  LSE is the log of the whole denominator.
 *     A row with a sink and no visible key therefore gives O = 0 and
 *     LSE = sigma_h in both masked-rows modes; a NaN or +inf score (the sink
 *     included) still makes the row NaN, and a sink of -inf adds nothing.
 *
 * Quantised key/value caches, from the same page (inputs k_scale and
 * v_scale, attributes k_quant_type, v_quant_type and kv_cache_bit_width = 8):
 * a cache element is a signed 8-bit integer and its value is that integer
 * times a float32 scale -- one scale for the whole cache (PER_TENSOR) or one
 * per (kv head, head-dim channel), kv_heads * head_dim of them (PER_CHANNEL).
 * The product is exact in double.
 *
 * Cache append ("com.microsoft.GroupQueryAttention": present_key /
 * present_value with past and present sharing one buffer; seqlens_k is the
 * total length including the new token; the int8 decode variant appends
 * int8-quantised rows): orc_append_rows writes each (batch, kv head)'s new
 * row at cache position L_b - 1, L_b the clamped length; nothing when
 * L_b = 0.  Reading for int8 caches (the pages give no rounding rule): the
 * code is x / scale rounded to the nearest integer, ties to even, saturated
 * to [-128, 127], computed in float32 -- the precision of the kernel that
 * takes the same decision.
 *
 * Precision: every product and sum is in double.  Inputs are read in their
 * storage type (float32, IEEE half or bfloat16 bit patterns) and widened
 * exactly to double.  The combine routine follows "Attention", section
 * "Accuracy at long key lengths" (split key ranges merged in range order).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2

typedef struct {
  int64_t offset, batch_stride, head_stride, row_stride; /* elements */
} orc_layout;

typedef struct {
  int32_t batch, heads, kv_heads, q_len, k_len, head_dim;
  int32_t dtype;          /* ORC_F32 / ORC_F16 / ORC_BF16 for Q, K, V */
  float scale;            /* 0 selects the float nearest 1/sqrt(head_dim) */
  int32_t causal;         /* 0 or 1 */
  int64_t causal_offset;  /* INT64_MIN selects k_len - q_len */
  int32_t masked_rows_zero;
  orc_layout q, k, v;
  orc_layout mask;        /* (batch, head, row) strides in floats; keys contiguous */
  int64_t seg_batch_stride;
  int32_t window_left;    /* -1: no window; else causal rows keep keys >= i + offset - window_left */
  int32_t causal_align;   /* 0: one offset; 1: batch b's offset is its clamped key length - q_len */
  int32_t k_lens_kind;    /* 0: k_lens are counts; 1: they are the last valid index (count - 1) */
  float softcap;          /* 0: off; > 0: scores are softcap * tanh(scale q.k / softcap) before the mask */
  int32_t smooth_softmax; /* 1: a sink logit joins each row's denominator (sigma = 0 unless head_sink) */
  const float* head_sink; /* NULL or float [heads]: per-head sink logits (turns the sink on) */
  int32_t kv_int8;        /* 1: K and V are int8 with scales; Q keeps dtype */
  int32_t kv_per_channel; /* 0: one scale each for K and V; 1: kv_heads * head_dim scales each */
  const float* k_scale;
  const float* v_scale;
} orc_problem;

/* ---- exact widening of the storage types --------------------------------- */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f + 1024), e - 25);     /* (1.f) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 is the upper half of a binary32. */
static double orc_bf16_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double orc_load(const void* base, int32_t dtype, int64_t idx) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)base)[idx];
    case ORC_F16: return orc_half_to_double(((const uint16_t*)base)[idx]);
    default: return orc_bf16_to_double(((const uint16_t*)base)[idx]);
  }
}

double orc_widen(int32_t dtype, uint32_t bits) {
  if (dtype == ORC_F32) {
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return dtype == ORC_F16 ? orc_half_to_double((uint16_t)bits) : orc_bf16_to_double((uint16_t)bits);
}

/* One key or value element: the stored value, or int8 times its scale. */
static double orc_load_kv(const orc_problem* p, const void* base, const float* scale, int64_t idx, int64_t g,
                          int64_t d) {
  if (!p->kv_int8) return orc_load(base, p->dtype, idx);
  const double s = (double)scale[p->kv_per_channel ? g * p->head_dim + d : 0];
  return (double)((const int8_t*)base)[idx] * s;
}

static int64_t orc_clamp(int64_t x, int64_t lo, int64_t hi) {
  return x < lo ? lo : (x > hi ? hi : x);
}

float orc_default_scale(int32_t head_dim) {
  return (float)(1.0 / sqrt((double)head_dim));
}

/* ---- one query row --------------------------------------------------------- */

typedef struct {
  const orc_problem* p;
  const void *q, *k, *v;
  const float* mask;
  const int32_t* seg;
  const int32_t* k_lens;
  const int64_t* rows;   /* (b, h, qi) triples, or NULL for every row in order */
  double* o;             /* [n_rows][head_dim] */
  double* lse;           /* [n_rows] */
  int64_t row_begin, row_end;
  int status;
} orc_job;

/* Structural visibility of key kk for row (b, qi): "Attention", section
 * "What it covers" (Masks row) and section "Special values"; segment rule from
 * "attention_forward ...", section "2) Phase 0". */
static int orc_visible(const orc_problem* p, const int32_t* seg, const int32_t* k_lens,
                       int64_t b, int64_t qi, int64_t kk) {
  int64_t kl = p->k_len;                        /* valid keys of this batch entry */
  if (k_lens) {
    kl = orc_clamp((int64_t)k_lens[b] + (p->k_lens_kind ? 1 : 0), 0, p->k_len);
    if (kk >= kl) return 0;
  }
  if (p->causal) {
    int64_t off;
    if (p->causal_align) off = kl - p->q_len;  /* right-aligned to this entry's live length */
    else off = p->causal_offset == INT64_MIN ? (int64_t)p->k_len - p->q_len : p->causal_offset;
    if (kk > qi + off) return 0;                /* after the row's diagonal key */
    if (p->window_left >= 0 && kk < qi + off - p->window_left) return 0;   /* left of the window */
  }
  if (seg) {
    int64_t start = orc_clamp((int64_t)seg[b * p->seg_batch_stride + qi], 0, p->k_len);
    if (kk < start) return 0;
  }
  return 1;
}

static void orc_row(const orc_job* j, int64_t b, int64_t h, int64_t qi,
                    double* s /* [k_len] */, unsigned char* vis /* [k_len] */,
                    double* o_row, double* lse_out) {
  const orc_problem* p = j->p;
  const int64_t D = p->head_dim;
  const int64_t g = h / (p->heads / p->kv_heads);          /* kv_h = h / q_per_group */
  const double scale = (double)(p->scale != 0.0f ? p->scale : orc_default_scale(p->head_dim));
  const int64_t qbase = p->q.offset + b * p->q.batch_stride + h * p->q.head_stride + qi * p->q.row_stride;

  /* Scores of the structurally visible keys: s = scale * (q . k) + mask. */
  int any_nan_or_pinf = 0;
  for (int64_t kk = 0; kk < p->k_len; ++kk) {
    vis[kk] = (unsigned char)orc_visible(p, j->seg, j->k_lens, b, qi, kk);
    if (!vis[kk]) continue;
    const int64_t kbase = p->k.offset + b * p->k.batch_stride + g * p->k.head_stride + kk * p->k.row_stride;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d)
      dot += orc_load(j->q, p->dtype, qbase + d) * orc_load_kv(p, j->k, p->k_scale, kbase + d, g, d);
    double sc = scale * dot;
    if (p->softcap > 0.0f) {
      const double cap = (double)p->softcap;
      sc = cap * tanh(sc / cap);
    }
    if (j->mask) {
      const int64_t mbase = p->mask.offset + b * p->mask.batch_stride + h * p->mask.head_stride +
                            qi * p->mask.row_stride;
      sc += (double)j->mask[mbase + kk];
    }
    s[kk] = sc;
    if (isnan(sc) || (isinf(sc) && sc > 0)) any_nan_or_pinf = 1;
  }

  /* Pass 1: classify the row and find the maximum over the keys with weight > 0
   * (and the sink logit, when there is one). */
  const double sigma = p->head_sink ? (double)p->head_sink[h] : 0.0;
  int sink_on = p->smooth_softmax || p->head_sink != NULL;
  if (sink_on && (isnan(sigma) || sigma == INFINITY)) any_nan_or_pinf = 1;   /* the sink is a score too */
  if (sink_on && sigma == -INFINITY) sink_on = 0;                               /* exp(-inf) adds nothing */
  if (any_nan_or_pinf) {
    for (int64_t d = 0; d < D; ++d) o_row[d] = NAN;
    *lse_out = NAN;
    return;
  }
  int any = 0;
  double m = -INFINITY;
  for (int64_t kk = 0; kk < p->k_len; ++kk) {
    if (!vis[kk] || !(s[kk] > -INFINITY)) continue;
    if (!any || s[kk] > m) m = s[kk];
    any = 1;
  }
  if (!any && !sink_on) {                      /* no visible key: NaN, or 0 under MaskedRows = Zero */
    for (int64_t d = 0; d < D; ++d) o_row[d] = p->masked_rows_zero ? 0.0 : NAN;
    *lse_out = -INFINITY;
    return;
  }
  if (sink_on && (!any || sigma > m)) m = sigma;

  /* Pass 2: l = sum of exp(s - m), increasing key order, then the sink term. */
  double l = 0.0;
  for (int64_t kk = 0; kk < p->k_len; ++kk)
    if (vis[kk] && s[kk] > -INFINITY) l += exp(s[kk] - m);
  if (sink_on) l += exp(sigma - m);

  /* Pass 3: O = sum of exp(s - m) V[k] / l; LSE = m + log(l). */
  for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
  for (int64_t kk = 0; kk < p->k_len; ++kk) {
    if (!vis[kk] || !(s[kk] > -INFINITY)) continue;
    const double w = exp(s[kk] - m);
    const int64_t vbase = p->v.offset + b * p->v.batch_stride + g * p->v.head_stride + kk * p->v.row_stride;
    for (int64_t d = 0; d < D; ++d) o_row[d] += w * orc_load_kv(p, j->v, p->v_scale, vbase + d, g, d);
  }
  for (int64_t d = 0; d < D; ++d) o_row[d] /= l;
  *lse_out = m + log(l);
}

static void* orc_worker(void* arg) {
  orc_job* j = (orc_job*)arg;
  const orc_problem* p = j->p;
  const int64_t nk = p->k_len > 0 ? p->k_len : 1;
  double* s = (double*)malloc(sizeof(double) * nk);
  unsigned char* vis = (unsigned char*)malloc(nk);
  if (!s || !vis) {
    free(s);
    free(vis);
    j->status = -2;
    return NULL;
  }
  for (int64_t r = j->row_begin; r < j->row_end; ++r) {
    int64_t b, h, qi;
    if (j->rows) {
      b = j->rows[3 * r];
      h = j->rows[3 * r + 1];
      qi = j->rows[3 * r + 2];
    } else {
      qi = r % p->q_len;
      h = (r / p->q_len) % p->heads;
      b = r / ((int64_t)p->q_len * p->heads);
    }
    orc_row(j, b, h, qi, s, vis, j->o + r * p->head_dim, j->lse + r);
  }
  free(s);
  free(vis);
  return NULL;
}

/*
 * orc_attn_rows: O and LSE of n_rows query rows.  rows = (b, h, qi) triples, or
 * NULL for all batch*heads*q_len rows in (b, h, qi) order.  o is [n_rows][head_dim],
 * lse is [n_rows], both double.  Returns 0, -1 on a bad argument, -2 on
 * allocation failure.
 */
int orc_attn_rows(const orc_problem* p, const void* q, const void* k, const void* v,
                  const float* mask, const int32_t* seg, const int32_t* k_lens,
                  int64_t n_rows, const int64_t* rows, double* o, double* lse, int32_t nthreads) {
  if (!p || p->batch < 0 || p->heads <= 0 || p->kv_heads <= 0 || p->heads % p->kv_heads ||
      p->q_len < 0 || p->k_len < 0 || p->head_dim <= 0 || n_rows < 0)
    return -1;
  if (n_rows == 0) return 0;
  if (!q || !o || !lse || (p->k_len > 0 && (!k || !v))) return -1;
  if (rows) {
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[3 * r] < 0 || rows[3 * r] >= p->batch || rows[3 * r + 1] < 0 ||
          rows[3 * r + 1] >= p->heads || rows[3 * r + 2] < 0 || rows[3 * r + 2] >= p->q_len)
        return -1;
  } else if (n_rows != (int64_t)p->batch * p->heads * p->q_len) {
    return -1;
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > n_rows) nthreads = (int32_t)n_rows;
  orc_job jobs[256];
  pthread_t tids[256];
  int started[256];
  for (int t = 0; t < nthreads; ++t) {
    orc_job* j = &jobs[t];
    j->p = p; j->q = q; j->k = k; j->v = v; j->mask = mask; j->seg = seg; j->k_lens = k_lens;
    j->rows = rows; j->o = o; j->lse = lse; j->status = 0;
    j->row_begin = n_rows * t / nthreads;
    j->row_end = n_rows * (t + 1) / nthreads;
    started[t] = (t > 0) && pthread_create(&tids[t], NULL, orc_worker, j) == 0;
  }
  orc_worker(&jobs[0]);
  int status = jobs[0].status;
  for (int t = 1; t < nthreads; ++t) {
    if (started[t]) pthread_join(tids[t], NULL);
    else orc_worker(&jobs[t]);
    if (jobs[t].status) status = jobs[t].status;
  }
  return status;
}

/*
 * orc_append_rows: the cache update that precedes a decode step.  For each
 * batch entry b with L_b = clamp(k_lens[b] + plus, 0, cap) >= 1 and each kv
 * head g, row L_b - 1 of the cache (BNSH: cache + b*bs + g*hs + row*rs) takes
 * new[(b * kv_heads + g) * D .. + D).  elem: 2 or 4 bytes when the cache holds
 * the new rows' type (a bit copy); 1 for an int8 cache, whose codes are the
 * float32-rounded x / scale (see the header), the new rows then being of
 * new_dtype (ORC_F32 / ORC_F16 / ORC_BF16) with scales per tensor (n_scale 1)
 * or per (g, d).  Returns 0, or -1 on a bad argument.
 */
int orc_append_rows(void* cache, int64_t bs, int64_t hs, int64_t rs, int32_t cap, int32_t batch,
                    int32_t kv_heads, int32_t D, int32_t elem, const void* new_rows, int32_t new_dtype,
                    const int32_t* k_lens, int32_t plus, const float* scale, int32_t per_channel) {
  if (!cache || !new_rows || !k_lens || cap < 0 || batch < 0 || kv_heads < 1 || D < 1) return -1;
  if (elem != 1 && elem != 2 && elem != 4) return -1;
  if (elem == 1 && !scale) return -1;
  for (int64_t b = 0; b < batch; ++b) {
    const int64_t L = orc_clamp((int64_t)k_lens[b] + plus, 0, cap);
    if (L < 1) continue;
    for (int64_t g = 0; g < kv_heads; ++g) {
      const int64_t src = (b * kv_heads + g) * D;
      const int64_t dst = b * bs + g * hs + (L - 1) * rs;
      if (elem == 1) {
        for (int64_t d = 0; d < D; ++d) {
          const float x = (float)orc_load(new_rows, new_dtype, src + d);
          const float s = scale[per_channel ? g * D + d : 0];
          float c = rintf(x / s);                       /* float32 division, ties to even */
          if (c > 127.0f) c = 127.0f;
          if (c < -128.0f) c = -128.0f;
          ((int8_t*)cache)[dst + d] = (int8_t)c;
        }
      } else {
        memcpy((char*)cache + dst * elem, (const char*)new_rows + src * elem, (size_t)D * elem);
      }
    }
  }
  return 0;
}

/*
 * orc_combine: merge per-range partial results of the same rows.
 * "Attention", section "Accuracy at long key lengths": each key range leaves a
 * partial (max, sum, accumulator) and a second pass merges them in range order.
 * Here a partial is (lse_r, O_r) with O_r already divided by its own sum, so
 * the whole row is O = sum_r exp(lse_r) O_r / sum_r exp(lse_r) and
 * LSE = log(sum_r exp(lse_r)), evaluated relative to M = max_r lse_r.
 * part_o is [rows][n_splits][head_dim] float, part_lse [rows][n_splits] float.
 * A range with lse = -inf is empty; any NaN or +inf lse makes the row NaN;
 * all ranges empty is a row with no visible key.
 */
int orc_combine(int32_t n_splits, int64_t rows, int32_t head_dim, const float* part_o,
                const float* part_lse, int32_t masked_rows_zero, double* o, double* lse) {
  if (n_splits < 0 || rows < 0 || head_dim <= 0) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    double* out = o + r * head_dim;
    int bad = 0, any = 0;
    double M = -INFINITY;
    for (int32_t i = 0; i < n_splits; ++i) {
      double x = (double)part_lse[r * n_splits + i];
      if (isnan(x) || (isinf(x) && x > 0)) bad = 1;
      else if (x > -INFINITY) {
        if (!any || x > M) M = x;
        any = 1;
      }
    }
    if (bad) {
      for (int32_t d = 0; d < head_dim; ++d) out[d] = NAN;
      lse[r] = NAN;
      continue;
    }
    if (!any) {
      for (int32_t d = 0; d < head_dim; ++d) out[d] = masked_rows_zero ? 0.0 : NAN;
      lse[r] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
    for (int32_t i = 0; i < n_splits; ++i) {
      double x = (double)part_lse[r * n_splits + i];
      if (!(x > -INFINITY)) continue;
      double w = exp(x - M);
      wsum += w;
      const float* src = part_o + (r * n_splits + i) * head_dim;
      for (int32_t d = 0; d < head_dim; ++d) out[d] += w * (double)src[d];
    }
    for (int32_t d = 0; d < head_dim; ++d) out[d] /= wsum;
    lse[r] = M + log(wsum);
  }
  return 0;
}
