// mla_decode.cu — split-KV paged MLA decode core for sm_103a (TMA + tcgen05 + TMEM).
//
// The operation ("[WIP][Attention] FlashAttn MLA": decode MQA in MLA; shapes from the
// kernel-test log in "[Attention] Blackwell FP8 MLA support with CUTLASS_MLA backend"):
// all query rows of a sequence (s_q new tokens x H heads, 576 wide) attend over one
// shared latent row per token; scores use all 576 columns, values the first 512.
//
// Orientation. The output of 128 query rows is 128 x 512 float32 = 256 KB, the whole
// tensor memory of an SM, and 128 query rows are 144 KB of bf16, most of shared
// memory. So the MMAs run "tokens on M": with a tile of 128 keys,
//     S^T[128 keys x RC rows] = Kt[128 x 576] . Q[RC x 576]^T          (QK^T)
//     O^T[512 dv x RC rows]  += Vt^T[512 x 128] . P^T[128 x RC]        (PV, 4 M-tiles)
// where RC (16, 32 or 64) query rows form one work unit. Both products read the same
// shared-memory copy layout of a key tile (a 64-column chunk is 128 rows x 128 bytes,
// 128-byte swizzle): as the K-major A operand of QK^T, and as the MN-major A operand
// of PV. S^T double-buffers in TMEM (2*RC columns) next to O^T (4*RC columns).
//
// Pipeline (one CTA per SM, persistent over the work units the scheduler sorted):
//   warp 0      key producer: Q of each unit, then the 9 key chunks (128 rows x 64
//               columns) of every tile into the K ring, one 16 KB slot per chunk. A K slot
//               is released as soon as its 4 QK^T MMAs complete, so key prefetch (the
//               HBM stream) never waits for the softmax.
//   warp 2      value producer: the 4 value chunk pairs (128 rows x 128 columns) of every
//               tile into the V ring (32 KB slots), fetched a second time for PV — they
//               were read from HBM for QK^T moments earlier and are L2-resident — so that
//               no slot lives from QK^T through the softmax to PV.
//   warp 1      MMA issuer (lane 0): QK(k+1) is issued before PV(k) so the tensor core
//               works while the softmax of tile k runs. The whole warp zeroes the value
//               rows past the sequence end in the last tile (the cache may hold NaN there
//               and 0 * NaN is NaN inside the MMA).
//   warps 4-7   softmax (one thread per key of the tile = one TMEM lane): scale, causal
//               mask, online softmax with a lazily-rescaled running max (the reference
//               max moves only when a score exceeds it by more than 2^8, so O^T is
//               rescaled rarely; the final normalisation uses the same reference, so the
//               result is exact), P^T to shared memory, epilogue (O^T / l -> output or
//               split partial plus LSE).
//   warps 8-11  FP8 cache only: E4M3 -> fp16 dequantisation (exact: each E4M3 value is
//               an fp16 value) of every chunk, from the producers' staging rings into the
//               K and V rings in the order the MMA consumes them, and bf16 -> fp16
//               conversion of Q. The FP8 path multiplies in fp16 with fp32
//               accumulation; kv_scale is folded into the score scale and the output.
//
// Every wait is bounded (mla_ptx.cuh): a stall sets the device error word and the CTA
// drains its in-flight copies and MMAs, frees its tensor memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "../../include/mla.h"

namespace mla {

constexpr int kKSlotBytes = 16384;   // one 64-column chunk of a tile: 128 rows x 128 B
constexpr int kVSlotBytes = 32768;   // two chunks: 128 value columns
constexpr int kHalfBytes = 8192;     // 64 rows x 128 B (one TMA box)
constexpr int kKStageBytes = 8192;   // FP8 chunk: 128 rows x 64 B
constexpr int kVStageBytes = 16384;  // FP8 chunk pair
constexpr int kStageHalf = 4096;     // 64 rows x 64 B (one TMA box)
constexpr int kChunksPerTile = 9;
constexpr int kPairsPerTile = 4;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kSoftmaxBar = 1;          // named barrier of the 4 softmax warps
constexpr int kSmemLimit = 232448;           // 227 KB per CTA
constexpr int kStaticBudget = 3072;          // static shared memory (barriers, scratch)

// Ring depths per configuration (RC query rows per unit, FP8 or bf16 cache), chosen to
// fill shared memory: Q (RC x 1152 B), the P^T buffers, then the rings.
template <int RC, bool FP8>
struct Cfg {
  static constexpr int kQBytes = RC * 1152;            // 9 chunks x RC rows x 128 B
  static constexpr int kPRow = RC * 2;                  // bytes of one P^T row (one key)
  static constexpr int kPBytes = 128 * kPRow;
  static constexpr int kNumP = RC == 64 ? 1 : 2;        // P^T buffers
  static constexpr uint32_t kPSwz = RC == 64 ? kSwizzle128 : RC == 32 ? kSwizzle64 : kSwizzle32;
  static constexpr int kTmemCols = RC == 64 ? 512 : RC == 32 ? 256 : 128;
  static constexpr int kThreads = FP8 ? 384 : 256;
  static constexpr int NK = FP8 ? (RC == 16 ? 4 : RC == 32 ? 3 : 2) : (RC == 16 ? 6 : 4);
  static constexpr int NV = FP8 ? 2 : (RC == 16 ? 3 : RC == 32 ? 3 : 2);
  static constexpr int NKS = FP8 ? (RC == 16 ? 4 : RC == 32 ? 3 : 2) : 0;
  static constexpr int NVS = FP8 ? (RC == 64 ? 1 : 2) : 0;
  static constexpr int kDynBytes = 1024 + kQBytes + kNumP * kPBytes + NK * kKSlotBytes +
                                   NV * kVSlotBytes + NKS * kKStageBytes + NVS * kVStageBytes;
  static_assert(kDynBytes + kStaticBudget <= kSmemLimit, "shared memory budget");
};

struct Unit {
  int b, g, tb, te, slot, L;
};

__device__ __forceinline__ Unit load_unit(const DecodeArgs& a, int u) {
  const int4 v = a.units[u];
  Unit r;
  r.b = v.x;
  r.g = v.y;
  r.tb = v.z & 0xFFFF;
  r.te = (int)((unsigned)v.z >> 16);
  r.slot = v.w;
  r.L = a.batch_info[r.b].z;
  return r;
}

// Swizzled byte offset of 16-byte unit `u` in row `row` of a P^T buffer whose rows are
// W bytes (W = 128/64/32 -> 128/64/32-byte swizzle, 8-row atoms of 8W bytes).
template <int W>
__device__ __forceinline__ uint32_t p_offset(int row, int u) {
  const uint32_t in_atom = (uint32_t)((row & 7) * W + 16 * u);
  const uint32_t swz = in_atom ^ ((((in_atom >> 7) & (W / 16 - 1))) << 4);
  return (uint32_t)(row >> 3) * (8 * W) + swz;
}

__device__ __forceinline__ int ordered(float x) {
  int k = __float_as_int(x);
  return k ^ ((k >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float unordered(int k) {
  return __int_as_float(k ^ ((k >> 31) & 0x7FFFFFFF));
}

// Two probabilities rounded to the MMA operand type (fp16 for the FP8 cache, else bf16).
template <bool FP8>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if (FP8) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Global row (page * P + offset) of the 64-key half `h` of tile `tile`, or -1 when the
// half lies wholly past the sequence end. A block-table entry outside the pool is
// flagged and mapped past the end of the tensor, where TMA reads zeros.
__device__ __forceinline__ int half_row(const DecodeArgs& a, const Unit& U, int tile, int h,
                                        uint32_t* err) {
  const int tok = tile * kTileTokens + 64 * h;
  if (tok >= U.L) return -1;
  int pg = a.block_table[(int64_t)U.b * a.MB + tok / a.P];
  if (pg < 0 || pg >= a.num_pages) {
    atomicOr(err, MLA_DEVERR_BLOCK_TABLE);
    pg = a.num_pages;
  }
  return pg * a.P + (tok % a.P);
}

// E4M3 -> fp16 of one 64-column chunk (128 rows) from a staging buffer laid out as two
// 64-row TMA boxes [half][64 rows][64 B] into the 128-byte-swizzled MMA layout
// [128 rows][128 B]. Rows at or past `valid` are written as zeros. 128 threads.
__device__ __forceinline__ void dequant_chunk(const uint8_t* src, uint8_t* dst, int valid, int t) {
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int uidx = it * 128 + t;          // 512 16-byte FP8 units per chunk
    const int row = uidx >> 2, q4 = uidx & 3;
    uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
    if (row < valid) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + (row >> 6) * kStageHalf +
                                                      (row & 63) * 64 + q4 * 16);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t hh[8];
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[k2] & 0xFFFFu), __NV_E4M3);
        __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[k2] >> 16), __NV_E4M3);
        hh[2 * k2] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
        hh[2 * k2 + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
      }
      o0 = make_uint4(hh[0], hh[1], hh[2], hh[3]);
      o1 = make_uint4(hh[4], hh[5], hh[6], hh[7]);
    }
    uint8_t* drow = dst + (row >> 3) * 1024 + (row & 7) * 128;
    *reinterpret_cast<uint4*>(drow + (((2 * q4) ^ (row & 7)) << 4)) = o0;
    *reinterpret_cast<uint4*>(drow + (((2 * q4 + 1) ^ (row & 7)) << 4)) = o1;
  }
}

template <int RC, bool FP8>
__global__ void __launch_bounds__(Cfg<RC, FP8>::kThreads, 1)
decode_kernel(const __grid_constant__ DecodeArgs a) {
  using C = Cfg<RC, FP8>;
  constexpr int NK = C::NK, NV = C::NV;
  constexpr int NKS = FP8 ? C::NKS : 1, NVS = FP8 ? C::NVS : 1;
  constexpr int NP = C::kNumP;

  extern __shared__ uint8_t dsmem_raw[];
  __shared__ __align__(8) uint64_t bar_kfull[NK], bar_kempty[NK], bar_vfull[NV], bar_vempty[NV];
  __shared__ __align__(8) uint64_t bar_ksfull[NKS], bar_ksempty[NKS], bar_vsfull[NVS], bar_vsempty[NVS];
  __shared__ __align__(8) uint64_t bar_qfull, bar_qready, bar_qempty;
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_s_empty[2], bar_p_full[NP], bar_pv[NP];
  __shared__ __align__(8) uint64_t bar_o_empty, bar_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ uint32_t abort_s;
  __shared__ float mref_s[RC], alpha_s[RC], tot_s[RC];
  __shared__ float wmax_s[4 * RC];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // carve the 1024-aligned dynamic region
  const uint32_t raw = smem_u32(dsmem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = dsmem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sP = sQ + C::kQBytes;
  const uint32_t sK = sP + NP * C::kPBytes;
  const uint32_t sV = sK + NK * kKSlotBytes;
  const uint32_t sKS = sV + NV * kVSlotBytes;
  const uint32_t sVS = sKS + (FP8 ? NKS * kKStageBytes : 0);
  uint8_t* gQ = gbase;
  uint8_t* gP = gbase + (sP - sQ);
  uint8_t* gK = gbase + (sK - sQ);
  uint8_t* gV = gbase + (sV - sQ);
  uint8_t* gKS = gbase + (sKS - sQ);
  uint8_t* gVS = gbase + (sVS - sQ);

  const uint32_t b_kfull = smem_u32(bar_kfull), b_kempty = smem_u32(bar_kempty);
  const uint32_t b_vfull = smem_u32(bar_vfull), b_vempty = smem_u32(bar_vempty);
  const uint32_t b_ksfull = smem_u32(bar_ksfull), b_ksempty = smem_u32(bar_ksempty);
  const uint32_t b_vsfull = smem_u32(bar_vsfull), b_vsempty = smem_u32(bar_vsempty);
  const uint32_t b_qfull = smem_u32(&bar_qfull), b_qready = smem_u32(&bar_qready);
  const uint32_t b_qempty = smem_u32(&bar_qempty);
  const uint32_t b_s_full = smem_u32(bar_s_full), b_s_empty = smem_u32(bar_s_empty);
  const uint32_t b_p_full = smem_u32(bar_p_full), b_pv = smem_u32(bar_pv);
  const uint32_t b_oempty = smem_u32(&bar_o_empty), b_drain = smem_u32(&bar_drain);
  volatile uint32_t* abort_flag = &abort_s;
  uint32_t* err = a.err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(b_kfull + 8 * i, FP8 ? 128 : 1);
      mbar_init(b_kempty + 8 * i, 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(b_vfull + 8 * i, FP8 ? 128 : 1);
      mbar_init(b_vempty + 8 * i, 1);
    }
    for (int i = 0; i < NKS; ++i) {
      mbar_init(b_ksfull + 8 * i, 1);
      mbar_init(b_ksempty + 8 * i, 128);
    }
    for (int i = 0; i < NVS; ++i) {
      mbar_init(b_vsfull + 8 * i, 1);
      mbar_init(b_vsempty + 8 * i, 128);
    }
    mbar_init(b_qfull, 1);
    mbar_init(b_qready, 128);
    mbar_init(b_qempty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_s_full + 8 * i, 1);
      mbar_init(b_s_empty + 8 * i, 128);
    }
    for (int i = 0; i < NP; ++i) {
      mbar_init(b_p_full + 8 * i, 128);
      mbar_init(b_pv + 8 * i, 1);
    }
    mbar_init(b_oempty, 128);
    mbar_init(b_drain, 1);
    abort_s = 0u;
    fence_mbarrier_init();
    tma_prefetch_desc(&a.tm_kv);
    tma_prefetch_desc(&a.tm_q);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  const int num_units = (int)a.hdr[1];
  const int R = a.R;

  auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
    return mbar_wait(bar, parity, abort_flag, err, MLA_DEVERR_TIMEOUT);
  };
  // A wait whose outcome the whole warp agrees on (any lane giving up -> all give up),
  // so warp-collective instructions after it never see a diverged warp.
  auto wait_warp = [&](uint32_t bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, wait(bar, parity)) != 0;
  };
  // The same for the 128 softmax threads, which also share a named barrier.
  auto wait_softmax = [&](uint32_t bar, uint32_t parity) -> bool {
    return !named_bar_or(kSoftmaxBar, 128, !wait(bar, parity));
  };
  // After an abort: wait (bounded, ignoring the abort flag) until the copies issued into
  // the last `depth` positions of a ring have landed, so no TMA writes after exit.
  auto drain_ring = [&](uint32_t full_bars, uint32_t pos, uint32_t depth) {
    volatile uint32_t no_abort = 0;
    const uint32_t first = pos > depth ? pos - depth : 0;
    for (uint32_t p = first; p < pos; ++p)
      mbar_wait(full_bars + 8 * (p % depth), (p / depth) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT);
  };

  if (warp == 0) {
    // ============================================================ key producer
    if (lane == 0) {
      uint32_t pos = 0, ucount = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++ucount) {
        const Unit U = load_unit(a, u);
        ok = wait(b_qempty, (ucount & 1) ^ 1);
        if (!ok) break;
        mbar_arrive_expect_tx(b_qfull, 9 * RC * 128);
        for (int c = 0; c < 9; ++c)
          tma_load_3d(sQ + c * RC * 128, &a.tm_q, b_qfull, c * 64, U.g * RC, U.b);
        for (int tile = U.tb; tile < U.te && ok; ++tile) {
          const int r0 = half_row(a, U, tile, 0, err), r1 = half_row(a, U, tile, 1, err);
          const int nh = r1 >= 0 ? 2 : 1;
          for (int c = 0; c < kChunksPerTile && ok; ++c, ++pos) {
            if (!FP8) {
              const uint32_t slot = pos % NK;
              ok = wait(b_kempty + 8 * slot, ((pos / NK) & 1) ^ 1);
              if (!ok) break;
              const uint32_t bar = b_kfull + 8 * slot, dst = sK + slot * kKSlotBytes;
              mbar_arrive_expect_tx(bar, nh * kHalfBytes);
              tma_load_2d(dst, &a.tm_kv, bar, c * 64, r0);
              if (nh == 2) tma_load_2d(dst + kHalfBytes, &a.tm_kv, bar, c * 64, r1);
            } else {
              const uint32_t slot = pos % NKS;
              ok = wait(b_ksempty + 8 * slot, ((pos / NKS) & 1) ^ 1);
              if (!ok) break;
              const uint32_t bar = b_ksfull + 8 * slot, dst = sKS + slot * kKStageBytes;
              mbar_arrive_expect_tx(bar, nh * kStageHalf);
              tma_load_2d(dst, &a.tm_kv, bar, c * 64, r0);
              if (nh == 2) tma_load_2d(dst + kStageHalf, &a.tm_kv, bar, c * 64, r1);
            }
          }
        }
      }
      if (!ok) {
        if (FP8) drain_ring(b_ksfull, pos, NKS);
        else drain_ring(b_kfull, pos, NK);
      }
    }
  } else if (warp == 2) {
    // ============================================================ value producer
    if (lane == 0) {
      uint32_t pos = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const Unit U = load_unit(a, u);
        for (int tile = U.tb; tile < U.te && ok; ++tile) {
          const int r0 = half_row(a, U, tile, 0, err), r1 = half_row(a, U, tile, 1, err);
          const int nh = r1 >= 0 ? 2 : 1;
          for (int j = 0; j < kPairsPerTile && ok; ++j, ++pos) {
            if (!FP8) {
              const uint32_t slot = pos % NV;
              ok = wait(b_vempty + 8 * slot, ((pos / NV) & 1) ^ 1);
              if (!ok) break;
              const uint32_t bar = b_vfull + 8 * slot, dst = sV + slot * kVSlotBytes;
              mbar_arrive_expect_tx(bar, 2 * nh * kHalfBytes);
              for (int sub = 0; sub < 2; ++sub) {
                tma_load_2d(dst + sub * kKSlotBytes, &a.tm_kv, bar, (2 * j + sub) * 64, r0);
                if (nh == 2)
                  tma_load_2d(dst + sub * kKSlotBytes + kHalfBytes, &a.tm_kv, bar, (2 * j + sub) * 64, r1);
              }
            } else {
              const uint32_t slot = pos % NVS;
              ok = wait(b_vsempty + 8 * slot, ((pos / NVS) & 1) ^ 1);
              if (!ok) break;
              const uint32_t bar = b_vsfull + 8 * slot, dst = sVS + slot * kVStageBytes;
              mbar_arrive_expect_tx(bar, 2 * nh * kStageHalf);
              for (int sub = 0; sub < 2; ++sub) {
                tma_load_2d(dst + sub * kKStageBytes, &a.tm_kv, bar, (2 * j + sub) * 64, r0);
                if (nh == 2)
                  tma_load_2d(dst + sub * kKStageBytes + kStageHalf, &a.tm_kv, bar, (2 * j + sub) * 64, r1);
              }
            }
          }
        }
      }
      if (!ok) {
        if (FP8) drain_ring(b_vsfull, pos, NVS);
        else drain_ring(b_vfull, pos, NV);
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    const uint32_t idesc_qk = make_idesc(128, RC, FP8 ? 0u : 1u, 0, 0);
    const uint32_t idesc_pv = make_idesc(128, RC, FP8 ? 0u : 1u, 1, 1);
    uint32_t kpos = 0, vpos = 0, gn = 0, ucount = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++ucount) {
      const Unit U = load_unit(a, u);
      const int T = U.te - U.tb;
      ok = wait_warp(FP8 ? b_qready : b_qfull, ucount & 1);
      if (!ok) break;
      tc_fence_after();
      for (int k = 0; k <= T && ok; ++k) {
        if (k < T) {
          // ---- scores of tile k into S buffer n&1
          const uint32_t n = gn + k, sb = n & 1;
          ok = wait_warp(b_s_empty + 8 * sb, ((n >> 1) & 1) ^ 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + sb * RC;
          for (int c = 0; c < kChunksPerTile && ok; ++c, ++kpos) {
            const uint32_t slot = kpos % NK;
            ok = wait_warp(b_kfull + 8 * slot, (kpos / NK) & 1);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = make_sdesc(sK + slot * kKSlotBytes + kk * 32, 16, 1024, kSwizzle128);
                const uint64_t bd = make_sdesc(sQ + c * RC * 128 + kk * 32, 16, 1024, kSwizzle128);
                umma_f16(d, ad, bd, idesc_qk, (c | kk) != 0);
              }
              umma_commit(b_kempty + 8 * slot);
            }
            __syncwarp();
          }
          if (!ok) break;
          if (lane == 0) {
            umma_commit(b_s_full + 8 * sb);
            if (k == T - 1) umma_commit(b_qempty);
          }
          __syncwarp();
        }
        if (k >= 1) {
          // ---- values of tile k-1 times P^T into O^T
          const uint32_t n = gn + k - 1, pb = n % NP;
          const bool first = (k == 1);
          ok = wait_warp(b_p_full + 8 * pb, (n / NP) & 1);
          if (!ok) break;
          if (first) ok = wait_warp(b_oempty, (ucount & 1) ^ 1);
          if (!ok) break;
          tc_fence_after();
          const int valid = U.L - (U.tb + k - 1) * kTileTokens;
          const int ksteps = valid >= kTileTokens ? 8 : (valid + 15) / 16;
          for (int j = 0; j < kPairsPerTile && ok; ++j, ++vpos) {
            const uint32_t slot = vpos % NV;
            ok = wait_warp(b_vfull + 8 * slot, (vpos / NV) & 1);
            if (!ok) break;
            if (!FP8 && valid < 16 * ksteps) {
              // zero the value rows [valid, 16*ksteps) of both chunks of this slot
              const int zrows = 16 * ksteps - valid;
              for (int i = lane; i < 2 * zrows * 8; i += 32) {
                const int sub = i / (zrows * 8);
                const int rem = i % (zrows * 8);
                const int row = valid + rem / 8;
                *reinterpret_cast<uint4*>(gV + slot * kVSlotBytes + sub * kKSlotBytes + row * 128 +
                                          (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
              for (int kk = 0; kk < ksteps; ++kk) {
                const uint64_t ad = make_sdesc(sV + slot * kVSlotBytes + kk * 2048, kKSlotBytes, 1024,
                                               kSwizzle128);
                const uint64_t bd = make_sdesc(sP + pb * C::kPBytes + kk * 16 * C::kPRow,
                                               8 * C::kPRow, 8 * C::kPRow, C::kPSwz);
                umma_f16(tmem + (2 + j) * RC, ad, bd, idesc_pv, !(first && kk == 0));
              }
              umma_commit(b_vempty + 8 * slot);
            }
            __syncwarp();
          }
          if (!ok) break;
          if (lane == 0) umma_commit(b_pv + 8 * pb);
          __syncwarp();
        }
      }
      gn += T;
    }
    // drain: every MMA issued has completed before tensor memory is released
    if (lane == 0) umma_commit(b_drain);
    __syncwarp();
    volatile uint32_t no_abort = 0;
    mbar_wait(b_drain, 0, &no_abort, err, MLA_DEVERR_TIMEOUT);
  } else if (warp >= 4 && warp < 8) {
    // ============================================================ softmax / epilogue
    const int w4 = warp - 4;
    const int t = w4 * 32 + lane;                       // key within the tile = TMEM lane
    const uint32_t lane_addr = (uint32_t)(w4 * 32) << 16;
    const float kvs = FP8 ? __ldg(a.kv_scale) : 1.0f;
    const float c_log2 = a.softmax_scale * kvs * kLog2e;
    uint32_t gn = 0;
    bool ok = true;
    float lsum[RC];
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const Unit U = load_unit(a, u);
      const int T = U.te - U.tb;
      if (t < RC) mref_s[t] = -INFINITY;
#pragma unroll
      for (int r = 0; r < RC; ++r) lsum[r] = 0.f;
      named_bar_sync(kSoftmaxBar, 128);
      const int row0 = U.g * RC;
      for (int k = 0; k < T && ok; ++k) {
        const uint32_t n = gn + k, sb = n & 1, pb = n % NP;
        ok = wait_softmax(b_s_full + 8 * sb, (n >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        float s[RC];
#pragma unroll
        for (int c = 0; c < RC / 16; ++c) tmem_ld16(tmem + lane_addr + sb * RC + 16 * c, s + 16 * c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(b_s_empty + 8 * sb);

        // keys visible to row r: L - s_q + 1 + i(r) when causal, else L
        const int j = (U.tb + k) * kTileTokens + t;
        bool need = false;
        const bool tail = (U.tb + k + 1) * kTileTokens > U.L - a.s_q + 1;   // any row may mask
#pragma unroll
        for (int r = 0; r < RC; ++r) {
          int nvis = U.L;
          if (tail && a.causal) nvis = min(U.L, U.L - a.s_q + 1 + (row0 + r) / a.H);
          const float x = j < nvis ? s[r] * c_log2 : -INFINITY;
          s[r] = x;
          need |= x > mref_s[r] + kRescaleLog2;
        }
        bool rescale = false;
        if (named_bar_or(kSoftmaxBar, 128, need)) {
#pragma unroll
          for (int r = 0; r < RC; ++r) {
            const int m = __reduce_max_sync(0xffffffffu, ordered(s[r]));
            if (lane == (r & 31)) wmax_s[w4 * RC + r] = unordered(m);
          }
          named_bar_sync(kSoftmaxBar, 128);
          if (t < RC) {
            const float old = mref_s[t];
            const float nm = fmaxf(fmaxf(old, fmaxf(wmax_s[t], wmax_s[RC + t])),
                                   fmaxf(wmax_s[2 * RC + t], wmax_s[3 * RC + t]));
            alpha_s[t] = nm == -INFINITY ? 1.f : ex2_approx(old - nm);
            mref_s[t] = nm;
          }
          named_bar_sync(kSoftmaxBar, 128);
#pragma unroll
          for (int r = 0; r < RC; ++r) lsum[r] *= alpha_s[r];
          rescale = k > 0;
        }
        // P^T row of this key, in registers until its buffer is free
        uint32_t pw[RC / 2];
#pragma unroll
        for (int r = 0; r < RC; r += 2) {
          const float p0 = s[r] == -INFINITY ? 0.f : ex2_approx(s[r] - mref_s[r]);
          const float p1 = s[r + 1] == -INFINITY ? 0.f : ex2_approx(s[r + 1] - mref_s[r + 1]);
          pw[r / 2] = pack2<FP8>(p0, p1);
          lsum[r] += p0;          // the normaliser sums the unrounded probabilities
          lsum[r + 1] += p1;
        }
        // the buffer's previous user, PV(n - NP), must have completed
        if (n >= (uint32_t)NP) {
          ok = wait_softmax(b_pv + 8 * pb, ((n / NP) - 1) & 1);
          if (!ok) break;
        }
        uint8_t* prow = gP + pb * C::kPBytes;
#pragma unroll
        for (int u16 = 0; u16 < C::kPRow / 16; ++u16)
          *reinterpret_cast<uint4*>(prow + p_offset<C::kPRow>(t, u16)) =
              make_uint4(pw[4 * u16], pw[4 * u16 + 1], pw[4 * u16 + 2], pw[4 * u16 + 3]);
        fence_proxy_async_smem();
        if (rescale) {
          // O^T holds tiles up to k-1 of this unit: wait for PV(n-1), then scale in place
          ok = wait_softmax(b_pv + 8 * ((n - 1) % NP), ((n - 1) / NP) & 1);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int jt = 0; jt < 4; ++jt) {
#pragma unroll
            for (int c = 0; c < RC / 16; ++c) {
              float o[16];
              const uint32_t ta = tmem + lane_addr + (2 + jt) * RC + 16 * c;
              tmem_ld16(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= alpha_s[16 * c + i];
              tmem_st16(ta, o);
            }
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(b_p_full + 8 * pb);
      }
      if (!ok) break;
      // ---- epilogue: wait for the unit's last PV
      {
        const uint32_t nl = gn + T - 1;
        ok = wait_softmax(b_pv + 8 * (nl % NP), (nl / NP) & 1);
        if (!ok) break;
      }
      tc_fence_after();
      // row sums: warp butterfly per row, then the 4 warp partials through shared memory
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        float v = lsum[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == (r & 31)) wmax_s[w4 * RC + r] = v;
      }
      named_bar_sync(kSoftmaxBar, 128);
      if (t < RC) tot_s[t] = (wmax_s[t] + wmax_s[RC + t]) + (wmax_s[2 * RC + t] + wmax_s[3 * RC + t]);
      named_bar_sync(kSoftmaxBar, 128);
      const bool direct = U.slot < 0;
#pragma unroll 1
      for (int jt = 0; jt < 4; ++jt) {
        const int dv = 128 * jt + t;
#pragma unroll
        for (int c = 0; c < RC / 16; ++c) {
          float o[16];
          tmem_ld16(tmem + lane_addr + (2 + jt) * RC + 16 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int r = 16 * c + i;
            const int rg = row0 + r;
            if (rg < R) {
              const float tot = tot_s[r];
              const float v = tot > 0.f ? o[i] * (kvs / tot) : 0.f;
              if (direct)
                a.out[((int64_t)U.b * R + rg) * kDV + dv] = __float2bfloat16_rn(v);
              else
                a.part_o[((int64_t)U.slot * R + rg) * kDV + dv] = v;
            }
          }
        }
      }
      if (t < RC && row0 + t < R) {
        const float tot = tot_s[t];
        const float l = tot > 0.f ? (mref_s[t] + __log2f(tot)) * kLn2 : -INFINITY;
        if (direct) a.lse[(int64_t)U.b * R + row0 + t] = l;
        else a.part_lse[(int64_t)U.slot * R + row0 + t] = l;
      }
      tc_fence_before();
      mbar_arrive(b_oempty);
      named_bar_sync(kSoftmaxBar, 128);
      gn += T;
    }
  } else if (FP8 && warp >= 8) {
    // ============================================================ FP8 dequant
    const int t = threadIdx.x - 256;                    // 0..127
    uint32_t kpos = 0, vpos = 0, ucount = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++ucount) {
      const Unit U = load_unit(a, u);
      const int T = U.te - U.tb;
      // Q: bf16 -> fp16 in place (same swizzled positions)
      ok = wait(b_qfull, ucount & 1);
      if (!ok) break;
      bool q_bad = false;
      for (int i = t; i < C::kQBytes / 16; i += 128) {
        uint4* p = reinterpret_cast<uint4*>(gQ + 16 * i);
        uint4 v = *p;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
          q_bad |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
          __half2 h = __floats2half2_rn(lo, hi);
          w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        *p = make_uint4(w[0], w[1], w[2], w[3]);
      }
      if (q_bad) atomicOr(err, MLA_DEVERR_Q_RANGE);
      fence_proxy_async_smem();
      mbar_arrive(b_qready);
      // chunks in the order the MMA consumes them: K(k) before V(k-1)
      for (int k = 0; k <= T && ok; ++k) {
        if (k < T) {
          const int valid = U.L - (U.tb + k) * kTileTokens;
          for (int c = 0; c < kChunksPerTile && ok; ++c, ++kpos) {
            const uint32_t ss = kpos % NKS, slot = kpos % NK;
            ok = wait(b_ksfull + 8 * ss, (kpos / NKS) & 1);
            if (!ok) break;
            ok = wait(b_kempty + 8 * slot, ((kpos / NK) & 1) ^ 1);
            if (!ok) break;
            dequant_chunk(gKS + ss * kKStageBytes, gK + slot * kKSlotBytes, valid, t);
            fence_proxy_async_smem();
            mbar_arrive(b_ksempty + 8 * ss);
            mbar_arrive(b_kfull + 8 * slot);
          }
        }
        if (k >= 1) {
          const int valid = U.L - (U.tb + k - 1) * kTileTokens;
          for (int j = 0; j < kPairsPerTile && ok; ++j, ++vpos) {
            const uint32_t ss = vpos % NVS, slot = vpos % NV;
            ok = wait(b_vsfull + 8 * ss, (vpos / NVS) & 1);
            if (!ok) break;
            ok = wait(b_vempty + 8 * slot, ((vpos / NV) & 1) ^ 1);
            if (!ok) break;
            for (int sub = 0; sub < 2; ++sub)
              dequant_chunk(gVS + ss * kVStageBytes + sub * kKStageBytes,
                            gV + slot * kVSlotBytes + sub * kKSlotBytes, valid, t);
            fence_proxy_async_smem();
            mbar_arrive(b_vsempty + 8 * ss);
            mbar_arrive(b_vfull + 8 * slot);
          }
        }
      }
    }
  }

  // ============================================================ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

template <int RC, bool FP8>
static cudaError_t prepare_one() {
  using C = Cfg<RC, FP8>;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<RC, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, decode_kernel<RC, FP8>);
  if (e != cudaSuccess) return e;
  if ((int)attr.sharedSizeBytes > kStaticBudget) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

template <int RC, bool FP8>
static cudaError_t launch_one(const DecodeArgs& a, int grid, cudaStream_t s) {
  using C = Cfg<RC, FP8>;
  decode_kernel<RC, FP8><<<grid, C::kThreads, C::kDynBytes, s>>>(a);
  return cudaGetLastError();
}

cudaError_t decode_prepare(int rc, bool fp8) {
  switch (rc * 2 + (fp8 ? 1 : 0)) {
    case 32: return prepare_one<16, false>();
    case 33: return prepare_one<16, true>();
    case 64: return prepare_one<32, false>();
    case 65: return prepare_one<32, true>();
    case 128: return prepare_one<64, false>();
    case 129: return prepare_one<64, true>();
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const DecodeArgs& a, int rc, bool fp8, int grid, cudaStream_t s) {
  switch (rc * 2 + (fp8 ? 1 : 0)) {
    case 32: return launch_one<16, false>(a, grid, s);
    case 33: return launch_one<16, true>(a, grid, s);
    case 64: return launch_one<32, false>(a, grid, s);
    case 65: return launch_one<32, true>(a, grid, s);
    case 128: return launch_one<64, false>(a, grid, s);
    case 129: return launch_one<64, true>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
