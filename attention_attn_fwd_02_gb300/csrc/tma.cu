// tma.cu -- TMA tensor-map encoding shared by the tensor-core prefill and the
// decode split pass.
#include <cudaTypedefs.h>

#include <mutex>

#include "tma.h"

namespace attn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

bool tma_map_bhsd(CUtensorMap* m, const void* base, int dtype, int D, int rows, int heads, int batch,
                  const Layout& l, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const char* ptr = static_cast<const char*>(base) + l.off * 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads, (cuuint64_t)batch};
  cuuint64_t rs = (cuuint64_t)l.rs * 2, hs = (cuuint64_t)l.hs * 2, bs = (cuuint64_t)l.bs * 2;
  // A stride is irrelevant when its extent is 1; give it a legal value.
  if (rows == 1 && rs == 0) rs = 16;
  if (heads == 1 && hs == 0) hs = 16;
  if (batch == 1 && bs == 0) bs = 16;
  cuuint64_t strides[3] = {rs, hs, bs};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                  const_cast<char*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tma_layout_ok_es(const void* base, const Layout& l, int rows, int heads, int batch, int es) {
  if (((uintptr_t)base + (uintptr_t)l.off * es) % 16) return false;
  auto ok = [es](int64_t stride, int extent) { return extent == 1 || (stride > 0 && (stride * es) % 16 == 0); };
  return ok(l.rs, rows) && ok(l.hs, heads) && ok(l.bs, batch) && l.rs * es < (1ll << 40) &&
         l.hs * es < (1ll << 40) && l.bs * es < (1ll << 40);
}

bool tma_layout_ok(const void* base, const Layout& l, int rows, int heads, int batch) {
  return tma_layout_ok_es(base, l, rows, heads, batch, 2);
}

bool tma_map_bhsd_u8(CUtensorMap* m, const void* base, int D, int rows, int heads, int batch, const Layout& l,
                     int box_rows) {
  auto fn = encode_fn();
  if (!fn || D > 128 || (D % 16) != 0) return false;
  const char* ptr = static_cast<const char*>(base) + l.off;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads, (cuuint64_t)batch};
  cuuint64_t rs = (cuuint64_t)l.rs, hs = (cuuint64_t)l.hs, bs = (cuuint64_t)l.bs;
  if (rows == 1 && rs == 0) rs = 16;
  if (heads == 1 && hs == 0) hs = 16;
  if (batch == 1 && bs == 0) bs = 16;
  cuuint64_t strides[3] = {rs, hs, bs};
  cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<char*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace attn
