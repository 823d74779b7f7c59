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
//   warp 0      TMA producer: Q of the unit, then key/value chunks into a ring of
//               32 KB slots in the order the MMA consumes them:
//               K(0) K(1) V(0) K(2) V(1) ... K(T-1) V(T-2) V(T-1); a K tile is 5
//               slots (chunk pairs {0,1}..{6,7}, {8}), a V tile 4 slots ({0,1}..{6,7}).
//               Values are fetched a second time for PV (they are L2-resident by then)
//               so that no slot has to live from QK^T through the softmax to PV.
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
//   warps 8-11  FP8 cache only: E4M3 -> fp16 dequantisation of every chunk (exact: each
//               E4M3 value is an fp16 value) from a staging ring into the MMA ring, and
//               bf16 -> fp16 conversion of Q. The FP8 path multiplies in fp16 with fp32
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

constexpr int kSlotBytes = 32768;    // ring slot: 2 chunks x 128 rows x 128 B
constexpr int kChunkBytes = 16384;   // 64 columns x 128 rows (bf16/fp16)
constexpr int kHalfBytes = 8192;     // 64 columns x 64 rows
constexpr int kStageBytes = 16384;   // FP8 staging slot: 2 chunks x 128 rows x 64 B
constexpr int kStageChunk = 8192;
constexpr int kStageHalf = 4096;
constexpr int kKSlots = 5;
constexpr int kVSlots = 4;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kSoftmaxBar = 1;          // named barrier of the 4 softmax warps
constexpr int kSmemLimit = 232448;           // 227 KB per CTA

template <int RC, bool FP8>
struct Cfg {
  static constexpr int kQBytes = RC * 1152;            // 9 chunks x RC rows x 128 B
  static constexpr int kPRow = RC * 2;                  // bytes of one P^T row (a key)
  static constexpr int kPBytes = 128 * kPRow;
  static constexpr uint32_t kPSwz = RC == 64 ? kSwizzle128 : RC == 32 ? kSwizzle64 : kSwizzle32;
  static constexpr int kTmemCols = RC == 64 ? 512 : RC == 32 ? 256 : 128;
  static constexpr int kThreads = FP8 ? 384 : 256;
  static constexpr int kFixed = kQBytes + 2 * kPBytes + 1024;   // + alignment slack
  static constexpr int kStatic = 4096;                            // static smem budget
  static constexpr int kNumStage = FP8 ? (RC == 64 ? 3 : 4) : 0;
  static constexpr int kNumSlots =
      (kSmemLimit - kStatic - kFixed - kNumStage * kStageBytes) / kSlotBytes;
  static constexpr int kDynBytes = kFixed + kNumSlots * kSlotBytes + kNumStage * kStageBytes;
  static_assert(kNumSlots >= 2, "ring too small");
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

template <int RC, bool FP8>
__global__ void __launch_bounds__(Cfg<RC, FP8>::kThreads, 1)
decode_kernel(const __grid_constant__ DecodeArgs a) {
  using C = Cfg<RC, FP8>;
  constexpr int NS = C::kNumSlots;
  constexpr int NST = FP8 ? C::kNumStage : 1;

  extern __shared__ uint8_t dsmem_raw[];
  __shared__ __align__(8) uint64_t bar_full[NS], bar_empty[NS];
  __shared__ __align__(8) uint64_t bar_sfull[NST], bar_sempty[NST];
  __shared__ __align__(8) uint64_t bar_qfull, bar_qready, bar_qempty;
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_s_empty[2], bar_p_full[2];
  __shared__ __align__(8) uint64_t bar_pv_done, bar_o_empty, bar_drain;
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
  const uint32_t sP = sQ + C::kQBytes;                 // two P^T buffers
  const uint32_t sRing = sP + 2 * C::kPBytes;
  const uint32_t sStage = sRing + NS * kSlotBytes;
  uint8_t* gQ = gbase;
  uint8_t* gP = gbase + C::kQBytes;
  uint8_t* gRing = gP + 2 * C::kPBytes;
  uint8_t* gStage = gRing + NS * kSlotBytes;

  const uint32_t b_full = smem_u32(bar_full), b_empty = smem_u32(bar_empty);
  const uint32_t b_sfull = smem_u32(bar_sfull), b_sempty = smem_u32(bar_sempty);
  const uint32_t b_qfull = smem_u32(&bar_qfull), b_qready = smem_u32(&bar_qready);
  const uint32_t b_qempty = smem_u32(&bar_qempty);
  const uint32_t b_s_full = smem_u32(bar_s_full), b_s_empty = smem_u32(bar_s_empty);
  const uint32_t b_p_full = smem_u32(bar_p_full);
  const uint32_t b_pv = smem_u32(&bar_pv_done), b_oempty = smem_u32(&bar_o_empty);
  const uint32_t b_drain = smem_u32(&bar_drain);
  volatile uint32_t* abort_flag = &abort_s;
  uint32_t* err = a.err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(b_full + 8 * i, FP8 ? 128 : 1);
      mbar_init(b_empty + 8 * i, 1);
    }
    for (int i = 0; i < NST; ++i) {
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_sempty + 8 * i, 128);
    }
    mbar_init(b_qfull, 1);
    mbar_init(b_qready, 128);
    mbar_init(b_qempty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_s_full + 8 * i, 1);
      mbar_init(b_s_empty + 8 * i, 128);
      mbar_init(b_p_full + 8 * i, 128);
    }
    mbar_init(b_pv, 1);
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

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      uint32_t pos = 0;
      uint32_t ucount = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++ucount) {
        const Unit U = load_unit(a, u);
        ok = wait(b_qempty, (ucount & 1) ^ 1);
        if (!ok) break;
        mbar_arrive_expect_tx(b_qfull, 9 * RC * 128);
        for (int c = 0; c < 9; ++c)
          tma_load_3d(sQ + c * RC * 128, &a.tm_q, b_qfull, c * 64, U.g * RC, U.b);
        const int T = U.te - U.tb;
        for (int k = 0; k <= T && ok; ++k) {
          for (int part = 0; part < 2 && ok; ++part) {
            // part 0: keys of tile k; part 1: values of tile k-1
            const bool isK = part == 0;
            if (isK && k == T) continue;
            if (!isK && k == 0) continue;
            const int tile = U.tb + (isK ? k : k - 1);
            int rowg[2];
            bool hv[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int tok = tile * kTileTokens + 64 * h;
              hv[h] = tok < U.L;
              rowg[h] = 0;
              if (hv[h]) {
                int pg = a.block_table[(int64_t)U.b * a.MB + tok / a.P];
                if (pg < 0 || pg >= a.num_pages) {
                  atomicOr(err, MLA_DEVERR_BLOCK_TABLE);
                  pg = a.num_pages;   // past the tensor end: TMA fills zeros
                }
                rowg[h] = pg * a.P + (tok % a.P);
              }
            }
            const int nh = hv[1] ? 2 : 1;
            const int nslots = isK ? kKSlots : kVSlots;
            for (int si = 0; si < nslots && ok; ++si, ++pos) {
              const int nsub = (isK && si == kKSlots - 1) ? 1 : 2;
              if (!FP8) {
                const uint32_t slot = pos % NS, ph = (pos / NS) & 1;
                ok = wait(b_empty + 8 * slot, ph ^ 1);
                if (!ok) break;
                mbar_arrive_expect_tx(b_full + 8 * slot, nsub * nh * kHalfBytes);
                for (int sub = 0; sub < nsub; ++sub)
                  for (int h = 0; h < nh; ++h)
                    tma_load_2d(sRing + slot * kSlotBytes + sub * kChunkBytes + h * kHalfBytes,
                                &a.tm_kv, b_full + 8 * slot, (2 * si + sub) * 64, rowg[h]);
              } else {
                const uint32_t ss = pos % NST, ph = (pos / NST) & 1;
                ok = wait(b_sempty + 8 * ss, ph ^ 1);
                if (!ok) break;
                mbar_arrive_expect_tx(b_sfull + 8 * ss, nsub * nh * kStageHalf);
                for (int sub = 0; sub < nsub; ++sub)
                  for (int h = 0; h < nh; ++h)
                    tma_load_2d(sStage + ss * kStageBytes + sub * kStageChunk + h * kStageHalf,
                                &a.tm_kv, b_sfull + 8 * ss, (2 * si + sub) * 64, rowg[h]);
              }
            }
          }
        }
      }
      if (!ok) {
        // drain: let every copy already issued land before the CTA can exit
        const uint32_t nring = FP8 ? NST : NS;
        const uint32_t first = pos > nring ? pos - nring : 0;
        const uint32_t fb = FP8 ? b_sfull : b_full;
        volatile uint32_t no_abort = 0;
        for (uint32_t p = first; p < pos; ++p)
          mbar_wait(fb + 8 * (p % nring), (p / nring) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    const uint32_t idesc_qk = make_idesc(128, RC, FP8 ? 0u : 1u, 0, 0);
    const uint32_t idesc_pv = make_idesc(128, RC, FP8 ? 0u : 1u, 1, 1);
    uint32_t pos = 0, gn = 0, ucount = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++ucount) {
      const Unit U = load_unit(a, u);
      const int T = U.te - U.tb;
      ok = wait_warp(FP8 ? b_qready : b_qfull, ucount & 1);
      if (!ok) break;
      tc_fence_after();
      for (int k = 0; k <= T && ok; ++k) {
        if (k < T) {
          const uint32_t n = gn + k, sb = n & 1;
          ok = wait_warp(b_s_empty + 8 * sb, ((n >> 1) & 1) ^ 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + sb * RC;
          for (int ks = 0; ks < kKSlots && ok; ++ks, ++pos) {
            const uint32_t slot = pos % NS;
            ok = wait_warp(b_full + 8 * slot, (pos / NS) & 1);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
              const int nsub = ks == kKSlots - 1 ? 1 : 2;
              for (int sub = 0; sub < nsub; ++sub) {
                const int chunk = 2 * ks + sub;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint64_t ad = make_sdesc(sRing + slot * kSlotBytes + sub * kChunkBytes + kk * 32,
                                                 16, 1024, kSwizzle128);
                  const uint64_t bd = make_sdesc(sQ + chunk * RC * 128 + kk * 32, 16, 1024, kSwizzle128);
                  umma_f16(d, ad, bd, idesc_qk, (ks | sub | kk) != 0);
                }
              }
              umma_commit(b_empty + 8 * slot);
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
          const uint32_t n = gn + k - 1, pb = n & 1;
          const bool first = (k == 1);
          ok = wait_warp(b_p_full + 8 * pb, (n >> 1) & 1);
          if (!ok) break;
          if (first) ok = wait_warp(b_oempty, (ucount & 1) ^ 1);
          if (!ok) break;
          tc_fence_after();
          const int valid = U.L - (U.tb + k - 1) * kTileTokens;
          const int ksteps = valid >= kTileTokens ? 8 : (valid + 15) / 16;
          for (int j = 0; j < kVSlots && ok; ++j, ++pos) {
            const uint32_t slot = pos % NS;
            ok = wait_warp(b_full + 8 * slot, (pos / NS) & 1);
            if (!ok) break;
            if (!FP8 && valid < 16 * ksteps) {
              // zero the value rows [valid, 16*ksteps) of both chunks of this slot
              const int zrows = 16 * ksteps - valid;
              for (int i = lane; i < 2 * zrows * 8; i += 32) {
                const int sub = i / (zrows * 8);
                const int rem = i % (zrows * 8);
                const int row = valid + rem / 8;
                const int u16 = rem % 8;
                *reinterpret_cast<uint4*>(gRing + slot * kSlotBytes + sub * kChunkBytes +
                                          row * 128 + u16 * 16) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
              for (int kk = 0; kk < ksteps; ++kk) {
                const uint64_t ad = make_sdesc(sRing + slot * kSlotBytes + kk * 2048,
                                               kChunkBytes, 1024, kSwizzle128);
                const uint64_t bd = make_sdesc(sP + pb * C::kPBytes + kk * 16 * C::kPRow,
                                               8 * C::kPRow, 8 * C::kPRow, C::kPSwz);
                umma_f16(tmem + (2 + j) * RC, ad, bd, idesc_pv, !(first && kk == 0));
              }
              umma_commit(b_empty + 8 * slot);
            }
            __syncwarp();
          }
          if (!ok) break;
          if (lane == 0) umma_commit(b_pv);
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
    uint32_t gn = 0, ucount = 0;
    bool ok = true;
    float lsum[RC];
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++ucount) {
      const Unit U = load_unit(a, u);
      const int T = U.te - U.tb;
      if (t < RC) mref_s[t] = -INFINITY;
#pragma unroll
      for (int r = 0; r < RC; ++r) lsum[r] = 0.f;
      named_bar_sync(kSoftmaxBar, 128);
      // keys visible to row r: L - s_q + 1 + i(r) when causal, else L
      const int row0 = U.g * RC;
      for (int k = 0; k < T && ok; ++k) {
        const uint32_t n = gn + k, sb = n & 1;
        ok = wait_softmax(b_s_full + 8 * sb, (n >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        float s[RC];
#pragma unroll
        for (int c = 0; c < RC / 16; ++c) tmem_ld16(tmem + lane_addr + sb * RC + 16 * c, s + 16 * c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(b_s_empty + 8 * sb);

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
        // P^T row of this key
        uint32_t pw[RC / 2];
#pragma unroll
        for (int r = 0; r < RC; r += 2) {
          const float p0 = s[r] == -INFINITY ? 0.f : ex2_approx(s[r] - mref_s[r]);
          const float p1 = s[r + 1] == -INFINITY ? 0.f : ex2_approx(s[r + 1] - mref_s[r + 1]);
          pw[r / 2] = pack2<FP8>(p0, p1);
          lsum[r] += p0;          // the normaliser sums the unrounded probabilities
          lsum[r + 1] += p1;
        }
        uint8_t* prow = gP + (n & 1) * C::kPBytes;
#pragma unroll
        for (int u16 = 0; u16 < C::kPRow / 16; ++u16)
          *reinterpret_cast<uint4*>(prow + p_offset<C::kPRow>(t, u16)) =
              make_uint4(pw[4 * u16], pw[4 * u16 + 1], pw[4 * u16 + 2], pw[4 * u16 + 3]);
        fence_proxy_async_smem();
        if (k > 0) {
          ok = wait_softmax(b_pv, (n - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          if (rescale) {
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
        }
        tc_fence_before();
        mbar_arrive(b_p_full + 8 * (n & 1));
      }
      if (!ok) break;
      // ---- epilogue
      ok = wait_softmax(b_pv, (gn + T - 1) & 1);
      if (!ok) break;
      tc_fence_after();
      float* red = reinterpret_cast<float*>(gP);          // both P^T buffers are idle now
#pragma unroll
      for (int r = 0; r < RC; r += 4)
        *reinterpret_cast<float4*>(red + t * RC + r) =
            make_float4(lsum[r], lsum[r + 1], lsum[r + 2], lsum[r + 3]);
      named_bar_sync(kSoftmaxBar, 128);
      if (t < RC) {
        float tot = 0.f;
        for (int x = 0; x < 128; ++x) tot += red[x * RC + t];
        tot_s[t] = tot;
      }
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
    uint32_t pos = 0, ucount = 0;
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
      for (int k = 0; k <= T && ok; ++k) {
        for (int part = 0; part < 2 && ok; ++part) {
          const bool isK = part == 0;
          if (isK && k == T) continue;
          if (!isK && k == 0) continue;
          const int tile = U.tb + (isK ? k : k - 1);
          const int valid = U.L - tile * kTileTokens;
          const int nslots = isK ? kKSlots : kVSlots;
          for (int si = 0; si < nslots && ok; ++si, ++pos) {
            const int nsub = (isK && si == kKSlots - 1) ? 1 : 2;
            const uint32_t ss = pos % NST, sph = (pos / NST) & 1;
            const uint32_t slot = pos % NS, ph = (pos / NS) & 1;
            ok = wait(b_sfull + 8 * ss, sph);
            if (!ok) break;
            ok = wait(b_empty + 8 * slot, ph ^ 1);
            if (!ok) break;
            const uint8_t* src = gStage + ss * kStageBytes;
            uint8_t* dst = gRing + slot * kSlotBytes;
            for (int sub = 0; sub < nsub; ++sub) {
#pragma unroll
              for (int it = 0; it < 4; ++it) {
                const int uidx = it * 128 + t;          // 512 16-byte FP8 units per chunk
                const int row = uidx >> 2, q4 = uidx & 3;
                uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
                if (row < valid) {
                  const uint4 v = *reinterpret_cast<const uint4*>(
                      src + sub * kStageChunk + (row >> 6) * kStageHalf + (row & 63) * 64 + q4 * 16);
                  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                  uint32_t h[8];
#pragma unroll
                  for (int k2 = 0; k2 < 4; ++k2) {
                    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                        (__nv_fp8x2_storage_t)(w[k2] & 0xFFFFu), __NV_E4M3);
                    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                        (__nv_fp8x2_storage_t)(w[k2] >> 16), __NV_E4M3);
                    h[2 * k2] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
                    h[2 * k2 + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
                  }
                  o0 = make_uint4(h[0], h[1], h[2], h[3]);
                  o1 = make_uint4(h[4], h[5], h[6], h[7]);
                }
                uint8_t* drow = dst + sub * kChunkBytes + (row >> 3) * 1024 + (row & 7) * 128;
                const int u0 = 2 * q4, u1 = 2 * q4 + 1;
                *reinterpret_cast<uint4*>(drow + ((u0 ^ (row & 7)) << 4)) = o0;
                *reinterpret_cast<uint4*>(drow + ((u1 ^ (row & 7)) << 4)) = o1;
              }
            }
            fence_proxy_async_smem();
            mbar_arrive(b_sempty + 8 * ss);
            mbar_arrive(b_full + 8 * slot);
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
  if ((int)attr.sharedSizeBytes > C::kStatic) return cudaErrorInvalidConfiguration;
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
