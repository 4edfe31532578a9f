// fattn_decode_paged_static: paged split-KV decode that allocates nothing.
//
// Some callers cannot allocate device memory for a workspace: plugins whose
// host (an inference server or another runtime) hands them only their input
// and output buffers, and code that runs inside a fixed device-memory budget
// owned by a pool it cannot draw from. This entry point runs the same decode
// kernels as fattn_decode_paged, but the split partials live in a file-scope
// device array of fixed size instead of a caller-provided workspace.
//
// The array is part of the library's device image, so every GPU that loads
// the library holds it (kStaticScratchBytes) until the process exits. In host
// code the array's name is only a host-side stand-in for the symbol, never a
// device address, so its device address is looked up with
// cudaGetSymbolAddress once per device (on the first call made with that
// device current) and cached.
#include "fattn.h"
#include "fattn_internal.h"

#include <atomic>

namespace {

constexpr size_t kStaticScratchBytes = FATTN_DECODE_STATIC_SCRATCH_BYTES;  // 32 MiB

__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::atomic<void*> g_scratch_device_addr[128];

// Device address of g_decode_scratch on the current device; nullptr on error.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  void* p = g_scratch_device_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress((void**)&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
  g_scratch_device_addr[dev].store(ptr, std::memory_order_release);
  return ptr;
}

}  // namespace

extern "C" fattn_status fattn_decode_paged_static(const void* q, const void* kcache, const void* vcache,
                                                  const int32_t* block_table, const int32_t* seqlens, int num_splits,
                                                  void* o, float* lse, int B, int Hq, int Hkv, int d, int page_size,
                                                  int max_pages_per_seq, int num_pages, float scale,
                                                  cudaStream_t stream) {
  // Argument checks without touching CUDA: fattn_decode_paged validates every
  // argument before it looks at the workspace, so a call with no workspace
  // returns FATTN_ERR_WORKSPACE exactly when everything else is valid.
  const fattn_status pre = fattn_decode_paged(q, kcache, vcache, block_table, seqlens, num_splits, o, lse, B, Hq, Hkv,
                                              d, page_size, max_pages_per_seq, num_pages, scale, nullptr, 0, stream);
  if (pre != FATTN_ERR_WORKSPACE) return pre;
  // Problems whose partials do not fit the fixed scratch are refused.
  if (fattn_decode_workspace_size(B, Hq, d, num_splits) > kStaticScratchBytes) return FATTN_ERR_WORKSPACE;
  void* scratch = scratch_address();
  if (!scratch) return FATTN_ERR_CUDA;
  // The scheduling counters that must start at zero are cleared by the decode
  // launch itself (cudaMemsetAsync on `stream`); every partial the merge reads
  // is written by this call's decode kernel.
  return fattn_decode_paged(q, kcache, vcache, block_table, seqlens, num_splits, o, lse, B, Hq, Hkv, d, page_size,
                            max_pages_per_seq, num_pages, scale, scratch, kStaticScratchBytes, stream);
}
