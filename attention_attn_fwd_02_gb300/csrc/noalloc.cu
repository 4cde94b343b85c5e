// noalloc.cu -- attn_decode_noalloc: the split-range decode with its scratch
// space in a fixed device array owned by this library, for callers that
// cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is not available or not
// allowed -- a host callback or a plugin handed only a stream, an allocator
// hook, a real-time loop that must not take the allocator's locks, a runtime
// that owns every byte of device memory and gives plugins none.  attn_decode
// asks its caller for a workspace; this entry point uses a file-scope
// __device__ array instead, so the caller passes only inputs and outputs.
//
// The array is kNoAllocScratchBytes (32 MiB) of device memory that every GPU
// on which this library is loaded holds until the process exits.  Its device
// address is looked up once per device (cudaGetSymbolAddress with that device
// current) on the first call made on that device: make that first call before
// any stream capture begins.  The address is kept per CUDA context, so a call
// after a cudaDeviceReset looks it up again in the device's new context.  In host code the array's name stands for a host
// shadow, not a device address, so only the looked-up pointer is ever passed
// to kernels.
//
// Every call shares the one array per device and it keeps the last call's
// contents.  The decode writes every partial result it later reads (an empty
// key range writes its empty marker), so nothing has to start at zero.  Calls
// whose GPU work overlaps (different streams, or different host threads) race
// on the array; serialise them, e.g. by issuing them on one stream.
#include "common.cuh"

namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

SymbolCache g_scratch_cache;

// Device address of the array on the current device and context (looked up
// once per device; again only if the device's context changed).
int scratch_address(void** out) {
  return symbol_address(g_scratch_cache, (const void*)&g_noalloc_scratch, out);
}

}  // namespace
}  // namespace attn

extern "C" {

size_t attn_decode_noalloc_max_scratch(void) { return attn::kNoAllocScratchBytes; }

int attn_decode_noalloc(const attn_problem* p, const void* q, const void* k_cache, const void* v_cache, void* o,
                        const float* mask, const int32_t* seg, const int32_t* k_lens, float* lse,
                        attn_stream stream) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_decode_workspace_size(p);
  if (need > attn::kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;  // beyond the fixed array
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = attn::scratch_address(&scratch);
    if (rc) return rc;
  }
  // need == 0: nothing to do (batch 0) or an invalid problem, which attn_decode reports.
  return attn_decode(p, q, k_cache, v_cache, o, mask, seg, k_lens, lse, scratch,
                     need > 0 ? attn::kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"
