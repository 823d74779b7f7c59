// mla_noalloc.cu — mla_decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin inside an inference engine
// whose plugin interface hands it only inputs and outputs, or a runtime that reserves
// all device memory up front through its own allocator and forbids other allocations
// (a stray cudaMalloc there can also stall every stream, because it may synchronise the
// device). mla_decode_noalloc serves them: the scratch memory mla_decode needs lives in
// a file-scope device array of this library, kNoAllocScratchBytes long, which every GPU
// that loads the library holds until the process exits.
//
// The array's name is only a host-side stand-in in host code, not a device address, so
// the address is looked up with cudaGetSymbolAddress once per device (the first call on
// that device, with that device current) and cached. Every call shares the one array:
// two calls that overlap on the GPU (on different streams, or from different threads)
// race on it. Nothing needs clearing between calls: the scheduler kernel writes every
// scratch word the later kernels read, in the same call. mla_decode_noalloc_check reads
// the device error word the last call left at the start of the array.
#include <atomic>
#include <cuda_runtime.h>
#include "mla_internal.h"
#include "../../include/mla.h"

namespace mla {
namespace {

constexpr size_t kNoAllocScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;   // 32 MiB
constexpr int kMaxDevs = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevs];

// The device address of g_noalloc_scratch on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevs) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace mla

extern "C" __attribute__((visibility("default"))) mla_status mla_decode_noalloc(
    const mla_decode_params* p, const void* q, const void* kv_cache, const int32_t* block_table,
    const int32_t* seq_lens, float softmax_scale, const float* kv_scale, void* out, float* lse,
    mla_stream_t stream) {
  if (p == nullptr) return MLA_ERR_INVALID_ARG;
  const size_t need = mla_decode_workspace_size(p, 0);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (need > mla::kNoAllocScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (mla::scratch_address(&scratch) != cudaSuccess) return MLA_ERR_CUDA;
  return mla_decode(p, q, kv_cache, block_table, seq_lens, softmax_scale, kv_scale, out, lse,
                    scratch, mla::kNoAllocScratchBytes, stream);
}

extern "C" __attribute__((visibility("default"))) mla_status mla_decode_noalloc_check(mla_stream_t stream,
                                                                                  uint32_t* bits) {
  void* scratch = nullptr;
  if (mla::scratch_address(&scratch) != cudaSuccess) return MLA_ERR_CUDA;
  return mla_decode_check(scratch, stream, bits);
}
