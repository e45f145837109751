// wan_text_embed_noalloc: the text projection (wan_text_embed) for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain scratch memory: code that runs while another
// component owns the whole device allocator (a host application that hands out only
// fixed buffers), code on a latency-critical path where an allocation could stall or
// fail, or plugins whose ABI only passes input and output pointers.  For them this entry
// point keeps the projection's scratch (the hidden activations between the two linear
// layers) in a statically sized device array that lives in this library's module for as
// long as the process has the library loaded on that device.
#include "kernels.h"

namespace wan {

// Maximum scratch: B * Lt * D elements of the hidden activations (2 bytes each in bf16,
// 4 bytes in fp32) must fit in this many bytes.
constexpr size_t kTextEmbedScratchBytes = 16u << 20;  // 16 MiB

}  // namespace wan

// The scratch array.  Every GPU that loads libwan holds one copy until the process exits.
static __device__ __align__(256) unsigned char g_text_embed_scratch[wan::kTextEmbedScratchBytes];

namespace {

// Device address of the scratch array on the current device.  In host code the array's
// name is only a host-side stand-in, so the kernels receive this address instead.  It is
// looked up on every call (cheap): an address cached per device ordinal would go stale
// if the caller reset the device and loaded the module again.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_text_embed_scratch) != cudaSuccess || p == nullptr) return WAN_ERR_CUDA;
  *out = p;
  return WAN_OK;
}

}  // namespace

extern "C" int wan_text_embed_noalloc(const void* text, const void* w1, const void* b1, const void* w2,
                                      const void* b2, void* ctx, int B, int Lt, int Ct, int D, int dtype,
                                      wan_stream_t stream) {
  if (dtype != WAN_BF16 && dtype != WAN_F32) return WAN_ERR_INVALID_ARG;
  if (B <= 0 || Lt <= 0 || Ct <= 0 || D <= 0) return WAN_ERR_INVALID_ARG;
  const size_t need = wan_text_embed_workspace_size(B, Lt, D, dtype);
  if (need == 0 || need > wan::kTextEmbedScratchBytes) return WAN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != WAN_OK) return st;
  return wan_text_embed(text, w1, b1, w2, b2, ctx, B, Lt, Ct, D, dtype, scratch, wan::kTextEmbedScratchBytes,
                        stream);
}

extern "C" size_t wan_text_embed_noalloc_max_bytes(void) { return wan::kTextEmbedScratchBytes; }
