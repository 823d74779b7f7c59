// mla_cache_write.cuh — one 8-value group of the paged cache write, shared by the
// cache-write kernel and the scheduler kernel of the fused cache-write + decode call.
//
// "[Attention] Blackwell FP8 MLA support with CUTLASS_MLA backend" (Purpose) adds an FP8
// KV cache: every latent value is stored as one E4M3 byte. Each token's 576-value row (512
// latent then 64 rope) goes to slot s = slot_mapping[t]: page s / P, row s % P. The bf16
// cache stores the bits; the FP8 cache stores e4m3_rne_satfinite(x / kv_scale), with the
// quotient an IEEE float32 division (spelled __fdiv_rn so that it stays correctly rounded)
// and CUDA's float -> e4m3 conversion in round-to-nearest-even, satfinite mode.
#pragma once
#include <cuda_fp8.h>
#include "mla_internal.h"
#include "../../include/mla.h"

namespace mla {

constexpr int kWriteGroupsPerToken = kDQK / 8;   // 72 groups of 8 values (16 bytes of bf16)

// Group c (0..71) of token t: 8 values in, 16 (bf16) or 8 (FP8) bytes out. A slot past the
// pool is skipped and flagged in *err; a negative slot (a padding token) is skipped.
template <bool FP8>
__device__ __forceinline__ void write_group(const uint4* __restrict__ latent, const uint4* __restrict__ rope,
                                            const int64_t* __restrict__ slots, int64_t t, int c,
                                            uint8_t* __restrict__ cache, int64_t total_slots, float scale,
                                            uint32_t* __restrict__ err) {
  const int64_t s = __ldg(slots + t);
  if (s < 0) return;
  if (s >= total_slots) {
    if (err != nullptr && c == 0) atomicOr(err, MLA_DEVERR_SLOT);
    return;
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

}  // namespace mla
