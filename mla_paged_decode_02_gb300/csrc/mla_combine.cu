// mla_combine.cu — merges the per-split partial outputs of split sequences.
//
// A sequence cut into key ranges (split-KV, flash-decoding) yields, per split s, the
// normalised partial output O_s and its log-sum-exp lse_s. The exact merge is
//   lse = log(sum_s exp(lse_s)),   out = sum_s exp(lse_s - lse) * O_s.
// A split with no visible key for a row (possible for causal s_q > 1) carries
// lse_s = -inf and weight 0.
//
// The scheduler cuts (sequence, row group) streams at CTA boundaries; each cut stream
// has `pieces` consecutive partial slots of RC rows. One warp per (cut stream, row):
// lane l owns output columns [16l, 16l+16), read as four float4 per piece (coalesced
// 2 KB rows). Persistent grid-stride loop over the list the scheduler wrote, so nothing
// launches per sequence. The kernel also checks, for the whole call, the block-table
// entries the decode read and the slots of a fused cache write (the error word was cleared
// by the scheduler, which ran before it).
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "../../include/mla.h"

namespace mla {

__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  const int lane = threadIdx.x & 31;
  // a fused cache write skipped slots outside the pool: report them
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, gstride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = gtid; i < a.w_n; i += gstride)
    if (a.w_slots[i] >= a.w_total_slots) atomicOr(a.err, MLA_DEVERR_SLOT);
  // block-table entries the decode read (the pages of each sequence up to its clamped
  // length) that lie outside the pool: the decode kernels read page 0 for them
  for (int64_t i = gtid; i < (int64_t)a.B * a.MB; i += gstride) {
    const int b = (int)(i / a.MB), j = (int)(i - (int64_t)b * a.MB);
    if ((int64_t)j * a.P < a.batch_info[b].z) {
      const int pg = a.block_table[i];
      if (pg < 0 || pg >= a.num_pages) atomicOr(a.err, MLA_DEVERR_BLOCK_TABLE);
    }
  }
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t tasks = (int64_t)a.hdr[2] * a.RC;
  for (int64_t task = warp; task < tasks; task += nwarps) {
    const int4 st = a.split_list[task / a.RC];
    const int r = (int)(task % a.RC);
    const int b = st.x, ns = st.z, base = st.w;
    const int rg = st.y * a.RC + r;          // row within the sequence
    if (rg >= a.R) continue;
    float m = -INFINITY;
    for (int s = 0; s < ns; ++s) m = fmaxf(m, a.part_lse[(int64_t)(base + s) * a.RC + r]);
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    float wsum = 0.f;
    for (int s = 0; s < ns; ++s) {
      const float ls = a.part_lse[(int64_t)(base + s) * a.RC + r];
      const float w = ls == -INFINITY ? 0.f : __expf(ls - m);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(
          a.part_o + ((int64_t)(base + s) * a.RC + r) * kDV) + lane * 4;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = src[k];
        acc[4 * k + 0] += w * v.x;
        acc[4 * k + 1] += w * v.y;
        acc[4 * k + 2] += w * v.z;
        acc[4 * k + 3] += w * v.w;
      }
    }
    const float inv = 1.f / wsum;
    uint32_t packed[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
      packed[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)b * a.R + rg) * kDV) + lane * 2;
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    if (lane == 0) a.lse[(int64_t)b * a.R + rg] = m + logf(wsum);
  }
}

// Plain stream order after the decode kernel: an early (programmatic) launch, whose
// blocks wait resident for the decode grid to finish, measured slower on long contexts.
cudaError_t launch_combine(const CombineArgs& a, int grid, cudaStream_t s) {
  combine_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
