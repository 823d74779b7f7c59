// umma_f8_probe.cu — test-only: one CTA runs the two 8-bit tcgen05 MMA operand layouts
// (kind::f8f6f4, E4M3 x E4M3, float32 accumulation) that the FP8-cache decode uses, on
// small known matrices, so that a test can compare them with torch.
//
// mode 0 ("scores"): D[128 x N] = A[128 x 128] . B[N x 128]^T
//   A: 128 rows x 128 E4M3 loaded by TMA as [16 row groups][2 chunks][8 rows][64 B] with
//      64-byte swizzle (the cache's key boxes): K-major, 8-row groups SBO = 1 KB apart
//   B: N rows x 128 E4M3 written by the threads in the same layout and swizzle
//   4 MMAs of K = 32: chunk c at +512 B, its second half at +32 B inside the atom.
// mode 1 ("values"): D[128 x N] = V^T . P,  V [64 keys x 128 columns], P [64 keys x N]
//   V: loaded by TMA as [8 key groups][2 chunks][8 keys][64 B], 64-byte swizzle: MN-major
//      A, the second 64-column chunk LBO = 512 B away, 8-key groups SBO = 1 KB apart
//   P: thread t writes key row t (N bytes, 64-byte swizzle for N = 64): MN-major B, 8-key
//      groups 512 B apart
//   2 MMAs of K = 32 keys.
// mode 2 ("values, P unswizzled"): as mode 1 with N in {16, 32, 64} and P written without
//   swizzle: key row t's N bytes as N / 16 core matrices of 16 B, [8-key group][core][8 keys]
//   [16 B]: MN-major B without swizzle, where the leading offset steps along K (8-key groups,
//   LBO = 8 N bytes) and the stride offset along MN (cores, SBO = 128 B).
// All waits are bounded; out-of-range modes return an error before launching.
#include <cstdint>
#include <cstring>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include "../../mla_paged_decode_02_gb300/csrc/mla_ptx.cuh"

using namespace mla;

namespace {

__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// byte offset of 16-byte unit u of row r in a [r/8][8][64 B] block sequence with the
// 64-byte swizzle (address bits [4,6) XOR bits [7,9))
__device__ __forceinline__ uint32_t sw64(uint32_t atom_base, int r, int u) {
  return atom_base + (uint32_t)(r & 7) * 64u + ((uint32_t)(u ^ ((r >> 1) & 3)) << 4);
}

}  // namespace

__global__ void __launch_bounds__(128, 1) f8_probe_kernel(const __grid_constant__ CUtensorMap tma_a,
                                                          const uint8_t* __restrict__ b_glob, int mode,
                                                          int n, float* __restrict__ d_out,
                                                          uint32_t* __restrict__ err) {
  extern __shared__ uint8_t raw[];
  __shared__ __align__(8) uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_s, abort_s;
  const uint32_t r0 = smem_u32(raw);
  const uint32_t base = (r0 + 1023u) & ~1023u;
  uint8_t* g = raw + (base - r0);
  const uint32_t sA = base;             // 16 KB
  const uint32_t sB = base + 16384;     // 16 KB
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

  const int t = threadIdx.x;
  if (mode == 0) {
    if (t == 0) {
      mbar_arrive_expect_tx(bt, 16384);
      tma_load_4d(sA, &tma_a, bt, 0, 0, 0, 0);
    }
    // B row t (t < n): 128 bytes = chunk 0 (units 0..3) and chunk 1 (units 4..7)
    if (t < n) {
      for (int u = 0; u < 8; ++u) {
        const uint4 v = *reinterpret_cast<const uint4*>(b_glob + t * 128 + u * 16);
        const uint32_t atom = (uint32_t)(t >> 3) * 1024u + (uint32_t)(u >> 2) * 512u;
        *reinterpret_cast<uint4*>(g + 16384 + sw64(atom, t, u & 3)) = v;
      }
    }
  } else if (mode == 2) {
    if (t == 0) {
      mbar_arrive_expect_tx(bt, 8192);
      tma_load_4d(sA, &tma_a, bt, 0, 0, 0, 0);
    }
    // P key row t (t < 64): n bytes, one 16-byte unit per core matrix
    if (t < 64) {
      for (int c = 0; c < n / 16; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(b_glob + t * n + c * 16);
        *reinterpret_cast<uint4*>(g + 16384 + (t >> 3) * (8 * n) + c * 128 + (t & 7) * 16) = v;
      }
    }
  } else {
    if (t == 0) {
      mbar_arrive_expect_tx(bt, 8192);
      tma_load_4d(sA, &tma_a, bt, 0, 0, 0, 0);
    }
    // P key row t (t < 64): n = 64 bytes, one 64-byte swizzled atom row
    if (t < 64) {
      for (int u = 0; u < 4; ++u) {
        const uint4 v = *reinterpret_cast<const uint4*>(b_glob + t * 64 + u * 16);
        *reinterpret_cast<uint4*>(g + 16384 + sw64((uint32_t)(t >> 3) * 512u, t, u)) = v;
      }
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  bool ok = mbar_wait(bt, 0, ab, err, 1u);
  if (ok && t == 0) {
    tc_fence_after();
    if (mode == 0) {
      const uint32_t idesc = make_idesc(128, (uint32_t)n, 0, 0, 0);
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t off = (uint32_t)(kk >> 1) * 512u + (uint32_t)(kk & 1) * 32u;
        const uint64_t ad = make_sdesc(sA + off, 16, 1024, kSwizzle64);
        const uint64_t bd = make_sdesc(sB + off, 16, 1024, kSwizzle64);
        mma_f8(tmem, ad, bd, idesc, kk > 0);
      }
    } else if (mode == 2) {
      const uint32_t idesc = make_idesc(128, (uint32_t)n, 0, 1, 1);
      for (int kk = 0; kk < 2; ++kk) {
        const uint64_t ad = make_sdesc(sA + kk * 4096, 512, 1024, kSwizzle64);
        const uint64_t bd = make_sdesc(sB + kk * 32 * n, 8 * n, 128, kSwizzleNone);
        mma_f8(tmem, ad, bd, idesc, kk > 0);
      }
    } else {
      const uint32_t idesc = make_idesc(128, 64, 0, 1, 1);
      for (int kk = 0; kk < 2; ++kk) {
        const uint64_t ad = make_sdesc(sA + kk * 4096, 512, 1024, kSwizzle64);
        const uint64_t bd = make_sdesc(sB + kk * 2048, 512, 512, kSwizzle64);
        mma_f8(tmem, ad, bd, idesc, kk > 0);
      }
    }
    umma_commit(bm);
  }
  __syncthreads();
  ok = mbar_wait(bm, 0, ab, err, 2u) && ok;
  tc_fence_after();
  if (ok) {
    float v[16];
    for (int c = 0; c < n / 16; ++c) {
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 16 * c, v);
      tmem_wait_ld();
      for (int i = 0; i < 16; ++i) d_out[(warp * 32 + lane) * n + 16 * c + i] = v[i];
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

// a [rows][128] byte matrix as [rows/8 groups][2 chunks][8 rows][64 B], one box of all of it
static int make_map(CUtensorMap* m, const void* ptr, uint64_t rows) {
  cuuint64_t dims[4] = {64, 8, 2, rows / 8};
  cuuint64_t strides[3] = {128, 64, 1024};
  cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(rows / 8)};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? 0
             : -1;
}

// mode 0: a [128 x 128] E4M3, b [n x 128] E4M3, n in {16, 32, 64}.
// mode 1: a = V [64 x 128] E4M3, b = P [64 x 64] E4M3 (n = 64).
// mode 2: a = V [64 x 128] E4M3, b = P [64 x n] E4M3, n in {16, 32, 64}.
// d [128 x n] float32. err: device uint32 (1 = TMA wait gave up, 2 = MMA wait gave up).
extern "C" __attribute__((visibility("default"))) int umma_f8_probe(int mode, int n, const void* a,
                                                                    const void* b, float* d,
                                                                    uint32_t* err, cudaStream_t s) {
  if (mode < 0 || mode > 2 || !a || !b || !d || !err) return -1;
  if (mode == 1 ? n != 64 : (n != 16 && n != 32 && n != 64)) return -1;
  if (!encoder()) return -2;
  CUtensorMap ta;
  if (make_map(&ta, a, mode == 0 ? 128 : 64)) return -3;
  const int smem = 32768 + 1024;
  cudaFuncSetAttribute(f8_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  f8_probe_kernel<<<1, 128, smem, s>>>(ta, static_cast<const uint8_t*>(b), mode, n, d, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
