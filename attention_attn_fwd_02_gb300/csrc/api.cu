// api.cu -- the C ABI of libattn.so: argument checks, planning and dispatch.
//
// Every entry point validates its arguments on the host, resolves the
// defaults (scale = float nearest 1/sqrt(head_dim), causal offset
// k_len - q_len: "Attention" (recursiveai.org OneGPU docs), section "What it
// covers"), picks a kernel from the dtype, head_dim and layout, and enqueues
// it on the caller's stream.  Nothing here allocates device memory or
// synchronises, except attn_device_status.
#include <math.h>
#include <string.h>

#include <atomic>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "prefill_tc.h"
#include "decode.h"

namespace attn {

// Sticky device status word: a kernel that gives up a bounded wait stores
// ATTN_ERR_DEVICE_TIMEOUT here; attn_device_status reads and clears it.
__device__ int g_status_word;

// One-shot fault for the bounded-wait tests (attn_test_inject): the next
// launch of a kernel that supports it takes it and clears it.
std::atomic<int> g_inject{ATTN_INJECT_NONE};

int take_injection() { return g_inject.exchange(ATTN_INJECT_NONE); }

namespace {

using PFN_ctx_current = CUresult (*)(CUcontext*);
using PFN_ctx_id = CUresult (*)(CUcontext, unsigned long long*);

// Driver entry points for the current context and its process-unique id,
// reached through the runtime (no libcuda link).  Null when unavailable.
void ctx_fns(PFN_ctx_current* cur, PFN_ctx_id* id) {
  static PFN_ctx_current f_cur = nullptr;
  static PFN_ctx_id f_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f_cur = reinterpret_cast<PFN_ctx_current>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f_id = reinterpret_cast<PFN_ctx_id>(p);
  });
  *cur = f_cur;
  *id = f_id;
}

// Id of the calling thread's current context; 0 when there is none yet or
// the driver cannot say.
unsigned long long current_ctx_id() {
  PFN_ctx_current cur;
  PFN_ctx_id id;
  ctx_fns(&cur, &id);
  CUcontext c = nullptr;
  unsigned long long v = 0;
  if (!cur || !id || cur(&c) != CUDA_SUCCESS || !c || id(c, &v) != CUDA_SUCCESS) return 0;
  return v;
}

}  // namespace

int symbol_address(SymbolCache& cache, const void* symbol, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(cache.mu);
  unsigned long long ctx = current_ctx_id();
  for (int i = 0; i < cache.n; ++i)
    if (cache.dev[i] == dev && cache.ctx[i] == ctx && ctx != 0) {
      *out = cache.ptr[i];
      return ATTN_OK;
    }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, symbol) != cudaSuccess || !ptr) return ATTN_ERR_CUDA;
  if (ctx == 0) ctx = current_ctx_id();   // the lookup above made the device's context current
  int slot = -1;
  for (int i = 0; i < cache.n; ++i)
    if (cache.dev[i] == dev) slot = i;    // a context of this device seen before: replace it
  if (slot < 0 && cache.n < SymbolCache::kSlots) slot = cache.n++;
  if (slot >= 0) {
    cache.dev[slot] = dev;
    cache.ctx[slot] = ctx;
    cache.ptr[slot] = ptr;
  }
  *out = ptr;
  return ATTN_OK;
}

namespace {

SymbolCache g_status_cache;

int status_ptr(int** out) {
  void* ptr = nullptr;
  const int rc = symbol_address(g_status_cache, (const void*)&g_status_word, &ptr);
  if (rc) return rc;
  *out = static_cast<int*>(ptr);
  return ATTN_OK;
}

size_t elem_size(int32_t dt) { return dt == ATTN_F32 ? 4 : 2; }

bool layout_ok(const attn_layout& l) {
  return l.offset >= 0 && l.batch_stride >= 0 && l.head_stride >= 0 && l.row_stride >= 0;
}

bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

// Checks the scalar fields; returns ATTN_OK or an error code.
int check_problem(const attn_problem* p) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (p->batch < 0 || p->heads < 1 || p->kv_heads < 1 || p->q_len < 0 || p->k_len < 0)
    return ATTN_ERR_INVALID_ARG;
  if (p->heads % p->kv_heads) return ATTN_ERR_INVALID_ARG;
  if (p->head_dim < 1 || p->head_dim > 256) return ATTN_ERR_INVALID_ARG;
  if (p->dtype != ATTN_F32 && p->dtype != ATTN_F16 && p->dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (p->dtype != ATTN_F32 && (p->head_dim & 1)) return ATTN_ERR_INVALID_ARG;  // half needs an even head_dim
  if (p->causal != 0 && p->causal != 1) return ATTN_ERR_INVALID_ARG;
  if (p->masked_rows != ATTN_MASKED_ROWS_NAN && p->masked_rows != ATTN_MASKED_ROWS_ZERO)
    return ATTN_ERR_INVALID_ARG;
  if (!(p->scale == p->scale) || isinf(p->scale)) return ATTN_ERR_INVALID_ARG;
  if (!layout_ok(p->q) || !layout_ok(p->k) || !layout_ok(p->v) || !layout_ok(p->o) || !layout_ok(p->mask))
    return ATTN_ERR_INVALID_ARG;
  if (p->seg_batch_stride < 0 || p->lse_batch_stride < 0 || p->lse_head_stride < 0) return ATTN_ERR_INVALID_ARG;
  if (p->window_left < -1 || (p->window_left >= 0 && !p->causal)) return ATTN_ERR_INVALID_ARG;
  if (p->causal_align != ATTN_CAUSAL_FIXED && p->causal_align != ATTN_CAUSAL_KLENS) return ATTN_ERR_INVALID_ARG;
  if (p->k_lens_kind != ATTN_KLENS_COUNT && p->k_lens_kind != ATTN_KLENS_LAST_INDEX) return ATTN_ERR_INVALID_ARG;
  if (!(p->softcap >= 0.0f) || isinf(p->softcap)) return ATTN_ERR_INVALID_ARG;
  if (p->smooth_softmax != 0 && p->smooth_softmax != 1) return ATTN_ERR_INVALID_ARG;
  if (p->head_sink && !aligned(p->head_sink, 4)) return ATTN_ERR_ALIGNMENT;
  if (p->kv_dtype != ATTN_KV_AS_Q && p->kv_dtype != ATTN_KV_INT8) return ATTN_ERR_INVALID_ARG;
  if (p->kv_scale_kind != ATTN_KV_SCALE_TENSOR && p->kv_scale_kind != ATTN_KV_SCALE_CHANNEL)
    return ATTN_ERR_INVALID_ARG;
  if (p->key_splits < 0) return ATTN_ERR_INVALID_ARG;
  if (p->kv_dtype == ATTN_KV_INT8) {
    if (!p->k_scale || !p->v_scale) return ATTN_ERR_INVALID_ARG;
    if (!aligned(p->k_scale, 4) || !aligned(p->v_scale, 4)) return ATTN_ERR_ALIGNMENT;
  }
  return ATTN_OK;
}

Problem resolve(const attn_problem* p, const void* q, const void* k, const void* v, void* o, const float* mask,
                const int32_t* seg, const int32_t* k_lens, float* lse, int* status) {
  Problem r;
  memset(&r, 0, sizeof r);
  r.B = p->batch;
  r.H = p->heads;
  r.G = p->kv_heads;
  r.Sq = p->q_len;
  r.Sk = p->k_len;
  r.D = p->head_dim;
  r.qpg = p->heads / p->kv_heads;
  r.dtype = p->dtype;
  r.scale = p->scale != 0.0f ? p->scale : (float)(1.0 / sqrt((double)p->head_dim));
  r.causal = p->causal;
  r.coff = p->causal_offset == ATTN_OFFSET_DEFAULT ? (int64_t)p->k_len - p->q_len : p->causal_offset;
  r.masked_zero = p->masked_rows == ATTN_MASKED_ROWS_ZERO;
  r.window = p->window_left;
  r.align_klens = p->causal_align == ATTN_CAUSAL_KLENS;
  r.klens_plus = p->k_lens_kind == ATTN_KLENS_LAST_INDEX ? 1 : 0;
  r.softcap = p->softcap;
  r.sink_on = (p->smooth_softmax || p->head_sink) ? 1 : 0;
  r.sink = p->head_sink;
  r.kv_int8 = p->kv_dtype == ATTN_KV_INT8;
  r.kv_per_channel = p->kv_scale_kind == ATTN_KV_SCALE_CHANNEL;
  r.k_scale = p->k_scale;
  r.v_scale = p->v_scale;
  r.q = {p->q.offset, p->q.batch_stride, p->q.head_stride, p->q.row_stride};
  r.k = {p->k.offset, p->k.batch_stride, p->k.head_stride, p->k.row_stride};
  r.v = {p->v.offset, p->v.batch_stride, p->v.head_stride, p->v.row_stride};
  r.o = {p->o.offset, p->o.batch_stride, p->o.head_stride, p->o.row_stride};
  r.m = {p->mask.offset, p->mask.batch_stride, p->mask.head_stride, p->mask.row_stride};
  r.seg_bs = p->seg_batch_stride;
  r.lse_bs = p->lse_batch_stride;
  r.lse_hs = p->lse_head_stride;
  r.Q = q;
  r.K = k;
  r.V = v;
  r.O = o;
  r.M = mask;
  r.seg = seg;
  r.klens = k_lens;
  r.lse = lse;
  r.status = status;
  return r;
}

int check_pointers(const attn_problem* p, const void* q, const void* k, const void* v, const void* o,
                   const float* mask, const int32_t* seg, const int32_t* k_lens, const float* lse) {
  const size_t es = elem_size(p->dtype);
  const size_t kv_es = p->kv_dtype == ATTN_KV_INT8 ? 1 : es;
  if (!q || !o) return ATTN_ERR_INVALID_ARG;
  if (p->k_len > 0 && (!k || !v)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, es) || !aligned(o, es) || (k && !aligned(k, kv_es)) || (v && !aligned(v, kv_es)))
    return ATTN_ERR_ALIGNMENT;
  if ((mask && !aligned(mask, 4)) || (seg && !aligned(seg, 4)) || (k_lens && !aligned(k_lens, 4)) ||
      (lse && !aligned(lse, 4)))
    return ATTN_ERR_ALIGNMENT;
  return ATTN_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Decode key-range plan: depends only on the shape ("Attention", section
// "Accuracy at long key lengths": ranges cut by the shape, merged in range
// order).  Ranges are a multiple of 32 keys, at least 128 keys, at most 8 of
// them a row: each range pays a fixed cost (its CTA's pipeline fill, Q load,
// four-warp merge and partial write), and on GB300 ranges of an eighth of
// the cache measured faster than sixteenths (the tail of unequal ranges
// grows less than the fixed costs shrink) and far faster than 32nds.
//
// int8 caches carry half the bytes per key, so those fixed costs weigh twice
// as much: their plan targets about 4096 ranges in all over (batch, kv head)
// pairs, at most 16 a row, each a multiple of the 64-key stage (measured
// against 2048, 8192 and 16384).
void decode_plan(const attn_problem* p, int* n_splits, int* split_len) {
  const int64_t Sk = p->k_len > 0 ? p->k_len : 1;
  if (p->kv_dtype == ATTN_KV_INT8) {
    const int64_t pairs = (int64_t)(p->batch > 0 ? p->batch : 1) * p->kv_heads;
    int64_t n = (4096 + pairs - 1) / pairs;
    n = n < 1 ? 1 : (n > 16 ? 16 : n);
    int64_t len = (Sk + n - 1) / n;
    len = (len + 63) / 64 * 64;
    if (len < 128) len = 128;
    *split_len = (int)len;
    *n_splits = (int)((Sk + len - 1) / len);
    return;
  }
  int64_t len = (Sk + 7) / 8;
  len = (len + 31) / 32 * 32;
  if (len < 128) len = 128;
  if (len > Sk) len = (Sk + 31) / 32 * 32;
  *split_len = (int)len;
  *n_splits = (int)((Sk + len - 1) / len);
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Prefill key-range plan ("Attention", section "Accuracy at long key
// lengths": ranges cut by the shape, at most 16, merged in range order).  A
// problem with fewer blocks of query rows than two per SM of a GB300 (304;
// 256 rows a block for head_dim <= 128, 128 above) and a long key axis gets
// ceil(304 / blocks) ranges, at most 16 and at most one per 1024 keys, so
// that each range's CTA has at least eight 128-key tiles to amortise its
// fixed cost; key_splits > 0 asks for a count instead.  Range lengths are a
// multiple of 128 keys (a key tile).
constexpr int kFillBlocks = 304;
constexpr int kMaxRanges = 16;

void fwd_plan(const attn_problem* p, int* n_splits, int* split_len) {
  const int64_t Sk = p->k_len;
  *n_splits = 1;
  *split_len = Sk > 0 ? (int)Sk : 1;
  if (Sk <= 0 || p->q_len <= 0 || p->batch <= 0) return;
  int64_t n;
  if (p->key_splits > 0) {
    n = p->key_splits < kMaxRanges ? p->key_splits : kMaxRanges;
  } else {
    const int rows = p->head_dim <= 128 ? 256 : 128;
    const int64_t blocks = (int64_t)((p->q_len + rows - 1) / rows) * p->heads * p->batch;
    if (blocks >= kFillBlocks) return;
    n = (kFillBlocks + blocks - 1) / blocks;
    n = n < kMaxRanges ? n : kMaxRanges;
    n = n < Sk / 1024 ? n : Sk / 1024;
  }
  if (n < 2) return;
  int64_t len = (Sk + n - 1) / n;
  len = (len + 127) / 128 * 128;
  *split_len = (int)len;
  *n_splits = (int)((Sk + len - 1) / len);
}

size_t decode_ws_bytes(const attn_problem* p, int n_splits) {
  const size_t rows = (size_t)p->batch * p->heads * p->q_len;
  return round256(rows * n_splits * p->head_dim * sizeof(float)) + round256(rows * n_splits * sizeof(float));
}

}  // namespace
}  // namespace attn

namespace attn {
namespace {
int decode_impl(const attn_problem* p, const void* q, const void* k_cache, const void* v_cache, void* o,
                const float* mask, const int32_t* seg, const int32_t* k_lens, float* lse, void* workspace,
                size_t workspace_bytes, attn_stream stream, const void* k_new, const void* v_new) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (p->q_len != 1) return ATTN_ERR_INVALID_ARG;
  if (p->batch == 0) return ATTN_OK;
  rc = check_pointers(p, q, k_cache, v_cache, o, mask, seg, k_lens, lse);
  if (rc) return rc;
  int n_splits = 1, split_len = 1;
  decode_plan(p, &n_splits, &split_len);
  const size_t need = decode_ws_bytes(p, n_splits);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return ATTN_ERR_ALIGNMENT;
  int* status = nullptr;
  rc = status_ptr(&status);
  if (rc) return rc;
  Problem r = resolve(p, q, k_cache, v_cache, o, mask, seg, k_lens, lse, status);
  r.k_new = k_new;
  r.v_new = v_new;
  const size_t rows = (size_t)p->batch * p->heads;
  Split s;
  s.n_splits = n_splits;
  s.split_len = split_len;
  s.part_o = static_cast<float*>(workspace);
  s.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        round256(rows * n_splits * p->head_dim * sizeof(float)));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int used = 0;
  rc = r.kv_int8 ? decode_q8_try(r, s, st, &used) : decode_fast_try(r, s, st, &used);
  if (rc) return rc;
  if (!used) {
    rc = from_cuda(launch_simt(r, s, st));
    if (rc) return rc;
  }
  return from_cuda(launch_combine(r, s, p->dtype, st));
}
}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

size_t attn_fwd_workspace_size(const attn_problem* p) {
  if (check_problem(p) != ATTN_OK) return 0;
  int n = 1, len = 1;
  fwd_plan(p, &n, &len);
  return n > 1 ? decode_ws_bytes(p, n) : 0;
}

int attn_fwd(const attn_problem* p, const void* q, const void* k, const void* v, void* o, const float* mask,
             const int32_t* seg, const int32_t* k_lens, float* lse, void* workspace, size_t workspace_bytes,
             attn_stream stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (p->batch == 0 || p->q_len == 0) return ATTN_OK;
  rc = check_pointers(p, q, k, v, o, mask, seg, k_lens, lse);
  if (rc) return rc;
  int n_splits = 1, split_len = 1;
  fwd_plan(p, &n_splits, &split_len);
  Split s{1, p->k_len > 0 ? p->k_len : 1, nullptr, nullptr};
  if (n_splits > 1) {
    const size_t need = decode_ws_bytes(p, n_splits);
    if (workspace && workspace_bytes >= need && aligned(workspace, 256)) {
      const size_t rows = (size_t)p->batch * p->heads * p->q_len;
      s.n_splits = n_splits;
      s.split_len = split_len;
      s.part_o = static_cast<float*>(workspace);
      s.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                            round256(rows * n_splits * p->head_dim * sizeof(float)));
    } else if (p->key_splits > 1) {
      return workspace && workspace_bytes >= need ? ATTN_ERR_ALIGNMENT : ATTN_ERR_WORKSPACE;
    }
  }
  int* status = nullptr;
  rc = status_ptr(&status);
  if (rc) return rc;
  Problem r = resolve(p, q, k, v, o, mask, seg, k_lens, lse, status);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int used = 0;
  rc = prefill_tc_try(r, s, st, &used);
  if (rc) return rc;
  if (!used) {
    rc = from_cuda(launch_simt(r, s, st));
    if (rc) return rc;
  }
  return s.n_splits > 1 ? from_cuda(launch_combine(r, s, p->dtype, st)) : ATTN_OK;
}

size_t attn_decode_workspace_size(const attn_problem* p) {
  if (check_problem(p) != ATTN_OK || p->q_len != 1) return 0;
  int n = 1, len = 1;
  decode_plan(p, &n, &len);
  return decode_ws_bytes(p, n);
}


int attn_decode(const attn_problem* p, const void* q, const void* k_cache, const void* v_cache, void* o,
                const float* mask, const int32_t* seg, const int32_t* k_lens, float* lse, void* workspace,
                size_t workspace_bytes, attn_stream stream) {
  return attn::decode_impl(p, q, k_cache, v_cache, o, mask, seg, k_lens, lse, workspace, workspace_bytes, stream,
                           nullptr, nullptr);
}

int attn_decode_append(const attn_problem* p, const void* q, const void* k_new, const void* v_new,
                       void* k_cache, void* v_cache, void* o, const float* mask, const int32_t* k_lens, float* lse,
                       void* workspace, size_t workspace_bytes, attn_stream stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (p->batch > 0 && (!k_new || !v_new || !k_lens || !k_cache || !v_cache)) return ATTN_ERR_INVALID_ARG;
  if (p->batch > 0 && p->k_len < 1) return ATTN_ERR_INVALID_ARG;
  const size_t es = elem_size(p->dtype);
  if ((k_new && !aligned(k_new, es)) || (v_new && !aligned(v_new, es))) return ATTN_ERR_ALIGNMENT;
  return attn::decode_impl(p, q, k_cache, v_cache, o, mask, nullptr, k_lens, lse, workspace, workspace_bytes,
                           stream, k_new, v_new);
}

int attn_combine(int32_t n_splits, int32_t rows, int32_t head_dim, const float* part_o, const float* part_lse,
                 int32_t out_dtype, void* o, int64_t o_row_stride, float* lse, int32_t masked_rows,
                 attn_stream stream) {
  if (n_splits < 0 || rows < 0 || head_dim < 1 || head_dim > 256 || o_row_stride < 0) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_F32 && out_dtype != ATTN_F16 && out_dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (masked_rows != ATTN_MASKED_ROWS_NAN && masked_rows != ATTN_MASKED_ROWS_ZERO) return ATTN_ERR_INVALID_ARG;
  if (rows == 0) return ATTN_OK;
  if (!o || (n_splits > 0 && (!part_o || !part_lse))) return ATTN_ERR_INVALID_ARG;
  if (!aligned(o, elem_size(out_dtype)) || (part_o && !aligned(part_o, 4)) || (part_lse && !aligned(part_lse, 4)) ||
      (lse && !aligned(lse, 4)))
    return ATTN_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return from_cuda(launch_combine_flat(n_splits, rows, head_dim, part_o, part_lse, out_dtype, o, o_row_stride, lse,
                                       masked_rows == ATTN_MASKED_ROWS_ZERO, st));
}

int attn_device_status(attn_stream stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int* ptr = nullptr;
  if (status_ptr(&ptr)) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess) return ATTN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess) return ATTN_ERR_CUDA;
  return v == 0 ? ATTN_OK : v;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported combination";
    case ATTN_ERR_ALIGNMENT: return "misaligned pointer";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    default: return "unknown status";
  }
}

int attn_probe_ex2(int32_t blocks, int32_t iters, float* sink, attn_stream stream) {
  if (blocks < 1 || iters < 1 || !sink || !aligned(sink, 4)) return ATTN_ERR_INVALID_ARG;
  return from_cuda(launch_ex2_probe(blocks, iters, sink, static_cast<cudaStream_t>(stream)));
}

int attn_test_inject(int32_t fault) {
  if (fault != ATTN_INJECT_NONE && fault != ATTN_INJECT_DROP_FIRST_COPY) return ATTN_ERR_INVALID_ARG;
  attn::g_inject.store(fault);
  return ATTN_OK;
}

int attn_version(void) { return 250; }

}  // extern "C"
