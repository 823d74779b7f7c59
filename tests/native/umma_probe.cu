// umma_probe.cu — test-only: one CTA runs the two tcgen05 MMA operand layouts the decode
// kernel relies on, on small known matrices, so a test can compare them with torch.
//
// mode 0 ("scores"): D[128 x N] = A[128 x 64] . B[N x 64]^T
//   A: 128 rows x 64 bf16 loaded by TMA (two 64-row boxes, 128-byte swizzle), K-major
//   B: N rows x 64 bf16 loaded by TMA (one N-row box, 128-byte swizzle), K-major
//   4 MMAs of K = 16, the start address advancing 32 bytes inside the swizzle atom.
// mode 1 ("values"): D[128 x N] = V^T . P,  V [128 keys x 128 dv], P [128 keys x N]
//   V: two 64-column chunks, each 128 rows x 128 B, 128-byte swizzle (TMA): MN-major A
//      with the second chunk LBO = 16 KB away and 8-key groups SBO = 1 KB apart
//   P: written by threads (thread = key row) with the swizzle of an N*2-byte row: MN-major B
//   8 MMAs of K = 16 keys, advancing 2 KB (A) and 16 rows (B).
// mode 2 ("scores, A in tensor memory"): D[128 x N] = A[128 x 64] . B[N x 64]^T with A
//   written by the threads into tensor memory (thread t = row t = TMEM lane t, two bf16
//   per 32-bit column, columns 64..95) and B as in mode 0; 4 MMAs of K = 16, the A
//   address advancing 8 columns.
// All waits are bounded; out-of-range modes return an error before launching.
#include <cstdint>
#include <cstring>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include "../../mla_paged_decode_02_gb300/csrc/mla_ptx.cuh"

using namespace mla;

template <int W>
__device__ __forceinline__ uint32_t p_off(int row, int u) {
  const uint32_t in_atom = (uint32_t)((row & 7) * W + 16 * u);
  const uint32_t swz = in_atom ^ ((((in_atom >> 7) & (W / 16 - 1))) << 4);
  return (uint32_t)(row >> 3) * (8 * W) + swz;
}

template <int N>
__global__ void __launch_bounds__(128, 1) probe_kernel(const __grid_constant__ CUtensorMap tma_a,
                                                       const __grid_constant__ CUtensorMap tma_b,
                                                       const __nv_bfloat16* __restrict__ p_glob,
                                                       int mode, float* __restrict__ d_out,
                                                       uint32_t* __restrict__ err) {
  extern __shared__ uint8_t raw[];
  __shared__ __align__(8) uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_s, abort_s;
  const uint32_t r0 = smem_u32(raw);
  const uint32_t base = (r0 + 1023u) & ~1023u;
  uint8_t* g = raw + (base - r0);
  const uint32_t sA = base;             // 32 KB
  const uint32_t sB = base + 32768;     // 16 KB
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bt = smem_u32(&bar_tma), bm = smem_u32(&bar_mma);
  if (threadIdx.x == 0) {
    mbar_init(bt, 1);
    mbar_init(bm, 1);
    abort_s = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_s), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;
  volatile uint32_t* ab = &abort_s;

  if (mode == 2) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bt, N * 128);
      tma_load_2d(sB, &tma_b, bt, 0, 0);
    }
    const int t = threadIdx.x;
    uint32_t w[32];
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(p_glob + t * 64);
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = arow[i];
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    tmem_st16u(lane_base + 64, w);
    tmem_st16u(lane_base + 80, w + 16);
    tmem_wait_st();
    tc_fence_before();
  } else if (mode == 0) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bt, 2 * 8192 + N * 128);
      tma_load_2d(sA, &tma_a, bt, 0, 0);
      tma_load_2d(sA + 8192, &tma_a, bt, 0, 64);
      tma_load_2d(sB, &tma_b, bt, 0, 0);
    }
  } else {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bt, 4 * 8192);
      for (int sub = 0; sub < 2; ++sub)
        for (int h = 0; h < 2; ++h) tma_load_2d(sA + sub * 16384 + h * 8192, &tma_a, bt, sub * 64, h * 64);
    }
    // thread t writes key row t of P with the row swizzle the decode kernel uses
    const int t = threadIdx.x;
    for (int u = 0; u < (N * 2) / 16; ++u) {
      uint4 v = *reinterpret_cast<const uint4*>(p_glob + t * N + u * 8);
      *reinterpret_cast<uint4*>(g + 32768 + p_off<N * 2>(t, u)) = v;
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  bool ok = mbar_wait(bt, 0, ab, err, 1u);
  if (ok && threadIdx.x == 0) {
    tc_fence_after();
    if (mode == 2) {
      const uint32_t idesc = make_idesc(128, N, 1, 0, 0);
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bd = make_sdesc(sB + kk * 32, 16, 1024, kSwizzle128);
        umma_f16_ts(tmem, tmem + 64 + kk * 8, bd, idesc, kk > 0);
      }
    } else if (mode == 0) {
      const uint32_t idesc = make_idesc(128, N, 1, 0, 0);
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = make_sdesc(sA + kk * 32, 16, 1024, kSwizzle128);
        const uint64_t bd = make_sdesc(sB + kk * 32, 16, 1024, kSwizzle128);
        umma_f16(tmem, ad, bd, idesc, kk > 0);
      }
    } else {
      const uint32_t idesc = make_idesc(128, N, 1, 1, 1);
      const uint32_t swz = N == 64 ? kSwizzle128 : N == 32 ? kSwizzle64 : kSwizzle32;
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = make_sdesc(sA + kk * 2048, 16384, 1024, kSwizzle128);
        const uint64_t bd = make_sdesc(sB + kk * 16 * N * 2, 8 * N * 2, 8 * N * 2, swz);
        umma_f16(tmem, ad, bd, idesc, kk > 0);
      }
    }
    umma_commit(bm);
  }
  __syncthreads();
  ok = mbar_wait(bm, 0, ab, err, 2u) && ok;
  tc_fence_after();
  if (ok) {
    float v[16];
    for (int c = 0; c < N / 16; ++c) {
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 16 * c, v);
      tmem_wait_ld();
      for (int i = 0; i < 16; ++i) d_out[(warp * 32 + lane) * N + 16 * c + i] = v[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

static int make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_c,
                    uint32_t box_r) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_c, box_r};
  cuuint32_t es[2] = {1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? 0
             : -1;
}

// mode 0: a [128 x 64] bf16, b [n x 64] bf16.  mode 1: a = V [128 x 128] bf16, b = P [128 x n].
// d [128 x n] float32. err: device uint32 (1 = TMA wait gave up, 2 = MMA wait gave up).
extern "C" __attribute__((visibility("default"))) int umma_probe(int mode, int n, const void* a,
                                                                 const void* b, float* d,
                                                                 uint32_t* err, cudaStream_t s) {
  if ((mode < 0 || mode > 2) || (n != 16 && n != 32 && n != 64) || !a || !b || !d || !err) return -1;
  if (!encoder()) return -2;
  CUtensorMap ta, tb;
  std::memset(&tb, 0, sizeof(tb));
  const __nv_bfloat16* pg = static_cast<const __nv_bfloat16*>(b);
  if (mode == 0) {
    if (make_map(&ta, a, 64, 128, 64, 64) || make_map(&tb, b, 64, n, 64, n)) return -3;
  } else if (mode == 2) {
    if (make_map(&tb, b, 64, n, 64, n)) return -3;
    ta = tb;
    pg = static_cast<const __nv_bfloat16*>(a);
  } else {
    if (make_map(&ta, a, 128, 128, 64, 64)) return -3;
    tb = ta;
  }
  const int smem = 32768 + 16384 + 1024;
  cudaError_t e;
  switch (n) {
    case 16:
      cudaFuncSetAttribute(probe_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      probe_kernel<16><<<1, 128, smem, s>>>(ta, tb, pg, mode, d, err);
      break;
    case 32:
      cudaFuncSetAttribute(probe_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      probe_kernel<32><<<1, 128, smem, s>>>(ta, tb, pg, mode, d, err);
      break;
    default:
      cudaFuncSetAttribute(probe_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      probe_kernel<64><<<1, 128, smem, s>>>(ta, tb, pg, mode, d, err);
  }
  e = cudaGetLastError();
  return e == cudaSuccess ? 0 : -4;
}
