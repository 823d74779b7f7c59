// mla_cache_write.cu — paged KV-cache write for MLA (bf16 copy or FP8 E4M3 quantise).
//
// "[Attention] Blackwell FP8 MLA support with CUTLASS_MLA backend" (Purpose) adds an
// FP8 KV cache to the decode path: every latent value is stored as one E4M3 byte. Each
// token's 576-value row (512 latent then 64 rope) goes to slot s = slot_mapping[t]:
// page s / P, row s % P. Quantisation is x / kv_scale in IEEE float32 (compiled without
// fast-math, and spelled __fdiv_rn so it stays correctly rounded) followed by CUDA's
// float -> e4m3 conversion in round-to-nearest-even, satfinite mode.
//
// Memory-bound scatter: one thread moves 8 values (16 bytes in, 16 or 8 bytes out);
// 72 threads cover one token, so the reads of a warp are contiguous.
#include <cuda_fp8.h>
#include "mla_internal.h"
#include "../../include/mla.h"

namespace mla {

template <bool FP8>
__global__ void __launch_bounds__(256) cache_write_kernel(
    const uint4* __restrict__ latent, const uint4* __restrict__ rope,
    const int64_t* __restrict__ slots, int32_t n_tokens, uint8_t* __restrict__ cache,
    int64_t total_slots, const float* __restrict__ kv_scale, uint32_t* __restrict__ err) {
  constexpr int kPerToken = kDQK / 8;   // 72 groups of 8 values
  const int64_t total = (int64_t)n_tokens * kPerToken;
  float scale = FP8 ? __ldg(kv_scale) : 1.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / kPerToken;
    const int c = (int)(i - t * kPerToken);
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= total_slots) {
      if (err != nullptr && c == 0) atomicOr(err, MLA_DEVERR_SLOT);
      continue;
    }
    const uint4 v = c < 64 ? __ldg(latent + t * 64 + c) : __ldg(rope + t * 8 + (c - 64));
    if (!FP8) {
      reinterpret_cast<uint4*>(cache + (size_t)s * kDQK * 2)[c] = v;
    } else {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t packed[2];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // two bf16 -> two float32 (exact) -> quotient -> two e4m3 bytes
        const float lo = __uint_as_float(w[k] << 16);
        const float hi = __uint_as_float(w[k] & 0xFFFF0000u);
        float2 q = make_float2(__fdiv_rn(lo, scale), __fdiv_rn(hi, scale));
        const __nv_fp8x2_storage_t b = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
        if (k & 1) packed[k >> 1] |= (uint32_t)b << 16;
        else packed[k >> 1] = (uint32_t)b;
      }
      reinterpret_cast<uint2*>(cache + (size_t)s * kDQK)[c] = make_uint2(packed[0], packed[1]);
    }
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
