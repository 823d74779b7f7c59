// mla_cache_write.cu — the paged KV-cache write kernel (bf16 copy or FP8 E4M3 quantise;
// the per-group arithmetic is in mla_cache_write.cuh).
//
// Memory-bound scatter: one thread moves 8 values (16 bytes in, 16 or 8 bytes out);
// 72 threads cover one token, so the reads of a warp are contiguous.
#include "mla_cache_write.cuh"

namespace mla {

template <bool FP8>
__global__ void __launch_bounds__(256) cache_write_kernel(
    const uint4* __restrict__ latent, const uint4* __restrict__ rope,
    const int64_t* __restrict__ slots, int32_t n_tokens, uint8_t* __restrict__ cache,
    int64_t total_slots, const float* __restrict__ kv_scale, uint32_t* __restrict__ err) {
  const int64_t total = (int64_t)n_tokens * kWriteGroupsPerToken;
  const float scale = FP8 ? __ldg(kv_scale) : 1.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / kWriteGroupsPerToken;
    write_group<FP8>(latent, rope, slots, t, (int)(i - t * kWriteGroupsPerToken), cache, total_slots, scale, err);
  }
}

cudaError_t launch_cache_write(const void* latent, const void* rope, const int64_t* slots,
                               int32_t n, void* cache, int64_t total_slots, bool fp8,
                               const float* kv_scale, uint32_t* err, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t work = (int64_t)n * (kDQK / 8);
  int64_t blocks = (work + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  if (fp8)
    cache_write_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(
        (const uint4*)latent, (const uint4*)rope, slots, n, (uint8_t*)cache, total_slots,
        kv_scale, err);
  else
    cache_write_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(
        (const uint4*)latent, (const uint4*)rope, slots, n, (uint8_t*)cache, total_slots,
        kv_scale, err);
  return cudaGetLastError();
}

}  // namespace mla
