// umma_pair_probe.cu — test-only: a cluster of two CTAs runs the CTA-pair tcgen05 MMA
// (cta_group::2, M = 256) in the two operand layouts the 128-row decode kernel uses, on
// small known matrices, so that a test can compare them with torch.
//
// mode 0 ("scores"): D[256 x 128] = A[256 x 64] . B[128 x 64]^T
//   CTA k holds A rows 128k..128k+127 (two 64-row TMA boxes, 128-byte swizzle, K-major)
//   and B rows 64k..64k+63 (one box); each CTA's tensor memory receives D rows
//   128k..128k+127 (lane = row) x all 128 columns. Each CTA waits for its own loads, then a
//   cluster barrier; the even CTA issues 4 MMAs of K = 16.
// mode 1 ("values"): D[256 x 128] = V^T . P with V [64 keys x 256] and P [64 keys x 128]
//   CTA k holds V columns 128k..128k+127 (two 64-column chunks, 128-byte swizzle:
//   MN-major A, LBO = the chunk stride, SBO = 1 KB per 8 keys) and P columns 64k..64k+63
//   (MN-major B, one 128-byte swizzle atom wide); 4 MMAs of K = 16 keys.
// mode 2: mode 0, but every TMA load (in either CTA) completes on the even CTA's mbarrier
//   (the cta_group::2 form of the TMA load), which is the only wait before the MMAs.
// Commits are multicast to the same mbarrier in both CTAs. All waits are bounded.
#include <cstdint>
#include <cstring>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include "../../mla_paged_decode_02_gb300/csrc/mla_ptx.cuh"

using namespace mla;

namespace {

__device__ __forceinline__ uint32_t ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void alloc2(uint32_t dst, uint32_t n) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst), "r"(n) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc2(uint32_t t, uint32_t n) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(t), "r"(n) : "memory");
}
__device__ __forceinline__ void mma2(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void commit2_both(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               :: "r"(bar), "h"((uint16_t)3) : "memory");
}
__device__ __forceinline__ void tma2d_to_leader(uint32_t dst, const CUtensorMap* m, uint32_t bar_cluster,
                                                int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1) : "memory");
}

__global__ void __launch_bounds__(128, 1) pair_probe_kernel(const __grid_constant__ CUtensorMap tma_a,
                                                            const __grid_constant__ CUtensorMap tma_b,
                                                            int mode, float* __restrict__ d_out,
                                                            uint32_t* __restrict__ err) {
  extern __shared__ uint8_t raw[];
  __shared__ __align__(8) uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_s, abort_s;
  const uint32_t r0 = smem_u32(raw);
  const uint32_t base = (r0 + 1023u) & ~1023u;
  const uint32_t sA = base;             // 16 KB
  const uint32_t sB = base + 16384;     // 8 KB
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ctarank();
  const uint32_t bt = smem_u32(&bar_tma), bm = smem_u32(&bar_mma);
  if (threadIdx.x == 0) {
    mbar_init(bt, 1);
    mbar_init(bm, 1);
    abort_s = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) alloc2(smem_u32(&tmem_s), 128);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();                   // both CTAs' barriers initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = tmem_s;
  volatile uint32_t* ab = &abort_s;

  if (threadIdx.x == 0) {
    if (mode == 0) {
      mbar_arrive_expect_tx(bt, 16384 + 8192);
      tma_load_2d(sA, &tma_a, bt, 0, 128 * rank);
      tma_load_2d(sA + 8192, &tma_a, bt, 0, 128 * rank + 64);
      tma_load_2d(sB, &tma_b, bt, 0, 64 * rank);
    } else if (mode == 1) {
      mbar_arrive_expect_tx(bt, 16384 + 8192);
      tma_load_2d(sA, &tma_a, bt, 128 * rank, 0);
      tma_load_2d(sA + 8192, &tma_a, bt, 128 * rank + 64, 0);
      tma_load_2d(sB, &tma_b, bt, 64 * rank, 0);
    } else {
      const uint32_t lb = map_rank(bt, 0);   // the even CTA's barrier
      if (rank == 0) mbar_arrive_expect_tx(bt, 2 * (16384 + 8192));
      tma2d_to_leader(sA, &tma_a, lb, 0, 128 * rank);
      tma2d_to_leader(sA + 8192, &tma_a, lb, 0, 128 * rank + 64);
      tma2d_to_leader(sB, &tma_b, lb, 0, 64 * rank);
    }
  }
  bool ok = true;
  if (mode != 2 || rank == 0) ok = mbar_wait(bt, 0, ab, err, 1u);
  if (mode != 2) {
    __syncthreads();
    cluster_sync_all();
  }
  if (ok && rank == 0 && threadIdx.x == 0) {
    tc_fence_after();
    if (mode == 1) {
      const uint32_t idesc = make_idesc(256, 128, 1, 1, 1);
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = make_sdesc(sA + kk * 2048, 8192, 1024, kSwizzle128);
        const uint64_t bd = make_sdesc(sB + kk * 2048, 1024, 1024, kSwizzle128);
        mma2(tmem, ad, bd, idesc, kk > 0);
      }
    } else {
      const uint32_t idesc = make_idesc(256, 128, 1, 0, 0);
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = make_sdesc(sA + kk * 32, 16, 1024, kSwizzle128);
        const uint64_t bd = make_sdesc(sB + kk * 32, 16, 1024, kSwizzle128);
        mma2(tmem, ad, bd, idesc, kk > 0);
      }
    }
    commit2_both(bm);
  }
  ok = mbar_wait(bm, 0, ab, err, 2u) && ok;
  tc_fence_after();
  if (ok) {
    float v[16];
    for (int c = 0; c < 8; ++c) {
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 16 * c, v);
      tmem_wait_ld();
      for (int i = 0; i < 16; ++i) d_out[(128 * rank + warp * 32 + lane) * 128 + 16 * c + i] = v[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();                   // no CTA leaves while its peer may still use it
  tc_fence_after();
  if (warp == 0) dealloc2(tmem, 128);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_c, uint32_t box_r) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_c, box_r};
  cuuint32_t es[2] = {1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? 0
             : -1;
}

}  // namespace

// mode 0/2: a [256 x 64] bf16, b [128 x 64] bf16.  mode 1: a = V [64 x 256], b = P [64 x 128].
// d [256 x 128] float32. err: device uint32 (1 = load wait gave up, 2 = MMA wait gave up).
extern "C" __attribute__((visibility("default"))) int umma_pair_probe(int mode, const void* a, const void* b,
                                                                      float* d, uint32_t* err, cudaStream_t s) {
  if (mode < 0 || mode > 2 || !a || !b || !d || !err) return -1;
  if (!encoder()) return -2;
  CUtensorMap ta, tb;
  if (mode == 1) {
    if (make_map(&ta, a, 256, 64, 64, 64) || make_map(&tb, b, 128, 64, 64, 64)) return -3;
  } else {
    if (make_map(&ta, a, 64, 256, 64, 64) || make_map(&tb, b, 64, 128, 64, 64)) return -3;
  }
  const int smem = 16384 + 8192 + 1024;
  if (cudaFuncSetAttribute(pair_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pair_probe_kernel, ta, tb, mode, d, err) == cudaSuccess ? 0 : -5;
}
