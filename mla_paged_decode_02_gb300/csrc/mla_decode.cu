// mla_decode.cu — split-KV paged MLA decode core for sm_103a (TMA + tcgen05 + TMEM).
//
// The operation ("[WIP][Attention] FlashAttn MLA", opening post: MLA decode runs as
// multi-query attention over the latent cache; shapes from the
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
// Pipeline (one CTA per SM, persistent over the contiguous range of work units the
// scheduler gave it). Every mbarrier ring slot has exactly one producer.
//   bf16 cache (256 threads):
//   warp 0      key producer (one thread): every key slot (KC chunks of a tile) is two 4D
//               TMA boxes, one per 64-row page half, landing directly in the swizzled
//               MMA layout.
//   warp 2      value producer: every value chunk pair as two TMA boxes, re-read from L2
//               so that no slot lives from QK^T through the softmax to PV; zeroes the rows
//               between the sequence end and the end of the last 16-key MMA step.
//   warp 1      QK^T issuer (one thread): Q of each unit (TMA), then per tile the S^T
//               buffer and every key slot in program order.
//   warp 3      PV issuer (one thread): per tile P^T, then the four value chunk pairs.
//   FP8 cache (384 threads): the MMAs read the E4M3 cache bytes as TMA landed them
//   (kind::f8f6f4), q and P entering as two E4M3 terms each (hi and lo).
//   16 or 32 rows:
//   warp 2      key-stage producer (one thread; the warp zeroes tail rows): each tile's
//               128 whole 576-byte rows into one of two stages, once the PV MMAs of the
//               tile that used it have completed; the stage serves both QK^T (keys) and
//               PV (values, the rows' first 512 bytes).
//   warps 8-11  each unit's Q, bf16 -> q' = q 2^e as E4M3 hi and lo in place, with the
//               row factors 2^-e for the softmax.
//   64 rows:
//   warps 8-11  one thread per key row: each unit's Q to fp16 in place; every raw E4M3
//               key position (TMA-staged) to fp16 in a tensor-memory key slot, read by
//               the QK^T MMAs as their A operand (kind::f16).
//   warp 2      raw value producer: 4-chunk E4M3 value stages, read by the PV MMAs.
//   warps 0, 1  PV and QK^T issuers.
//   both:
//   warps 4-7   softmax (one thread per key of the tile = one TMEM lane): scale, causal
//               mask, online softmax with a lazily-rescaled running max (the reference
//               max moves only when a score exceeds it by more than 2^8 (FP8: 2^4), so
//               O^T is rescaled rarely; the final normalisation uses the same reference,
//               so the result is exact), P^T to shared memory; epilogue (O^T / l ->
//               output or split partial plus LSE).
//
// Every wait is bounded (mla_ptx.cuh): a stall sets the device error word and the CTA
// waits for its in-flight copies and MMAs, frees its tensor memory and exits. Value rows
// past the sequence end are written as zeros by the loaders (the cache may hold NaN
// there and 0 * NaN is NaN inside the MMA).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <type_traits>
#include "mla_internal.h"
#include "mla_pages.cuh"
#include "mla_ptx.cuh"
#include "../../include/mla.h"

namespace mla {

constexpr int kChunkBytes = 16384;   // one 64-column chunk of a tile: 128 rows x 128 B
constexpr int kVSlotBytes = 32768;   // two chunks: 128 value columns
constexpr int kPairsPerTile = 4;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kSoftmaxBar = 1;          // named barrier of the 4 softmax warps
constexpr uint32_t kKeyDqBar = 2;            // FP8: warps 8-11 (Q, and keys with 64 rows)
constexpr int kKeyDqThreads = 128;
constexpr int kSmemLimit = 232448;           // 227 KB per CTA
constexpr int kStaticBudget = 3072;          // static shared memory (barriers, scratch)

// Ring depths per configuration (RC query rows per unit, FP8 or bf16 cache), chosen to
// fill shared memory: Q (RC x 1152 B), the P^T buffers, then the rings. A key slot holds
// KC chunks: every slot costs the issuing thread one barrier wait, one proxy fence and
// one commit, which are worth amortising over several chunks.
template <int RC, bool FP8>
struct Cfg {
  static constexpr int kQBytes = RC * 1152;            // 9 chunks x RC rows x 128 B
  static constexpr int kPRow = RC * 2;                  // bytes of one P^T row (one key)
  static constexpr int kPBytes = 128 * kPRow;
  static constexpr int kNumP = FP8 && RC == 64 ? 1 : 2;  // P^T buffers
  static constexpr uint32_t kPSwz = RC == 64 ? kSwizzle128 : RC == 32 ? kSwizzle64 : kSwizzle32;
  static constexpr int kTmemCols = FP8 || RC == 64 ? 512 : RC == 32 ? 256 : 128;
  static constexpr int kThreads = FP8 ? 384 : 256;
  static constexpr int kPvWarp = FP8 ? 0 : 3;           // warp of the PV issuing thread
  static constexpr int KC = RC == 64 ? 1 : 3;            // key chunks per K ring slot
  static constexpr int kKSlotBytes = KC * kChunkBytes;
  static constexpr int kSlotsPerTile = 9 / KC;
  // Ring layouts, as strides of the MMA operand descriptors. bf16 (TMA boxes): a key slot
  // is [16 row groups][KC chunks][8 rows x 128 B], a value slot [16 groups][2 chunks][...].
  // FP8 with 64 rows: the keys dequantised into tensor memory (below).
  static constexpr uint32_t kKGroupStride = FP8 ? 1024 : KC * 1024;    // key operand SBO
  static constexpr uint32_t kKChunkStride = FP8 ? kChunkBytes : 1024;
  static constexpr uint32_t kVChunkStride = FP8 ? kChunkBytes : 1024;  // value operand LBO
  static constexpr uint32_t kVGroupStride = FP8 ? 1024 : 2048;         // value operand SBO
  // FP8 with 64 rows: the dequantised key slots live in tensor memory after S^T (2 RC
  // columns) and O^T (4 RC columns), KC chunks x 32 columns each (two fp16 per column)
  static constexpr int kKTmemBase = 6 * RC;
  static constexpr int kKTmemSlotCols = KC * 32;
  static constexpr int NK = FP8 ? (RC == 32 ? 3 : 4) : (RC < 64 ? 2 : 3);
  // FP8 raw staging (E4M3 as TMA landed it, 64-byte swizzle). With 16 or 32 rows a key stage
  // is a tile's 128 whole 576-byte rows (two 64-row boxes, 72 KB), which feeds all of its
  // TMEM key positions and, its first 512 bytes per row, the PV MMAs as well; two stages.
  // 64 rows (whose Q and P^T leave no room for that) keep 1-chunk key stages and separate
  // 4-chunk value stages (256 value columns of the tile's rows, 32 KB).
  static constexpr bool kRawRows = FP8 && RC <= 32;
  static constexpr int NV = FP8 ? 1 : RC == 16 ? 3 : 2;     // bf16 value slots (FP8: none)
  static constexpr int kKRawChunks = kRawRows ? 9 : KC;     // chunks of a row per raw key box
  static constexpr int kKStageBytes = kKRawChunks * 8192;   // 2 halves x 64 rows x chunks x 64 B
  static constexpr int kKPosPerStage = kRawRows ? kSlotsPerTile : 1;   // TMEM key positions per stage
  static constexpr int kVRawChunks = 4;                     // chunks of a row per raw value box
  static constexpr int kVStage = kVRawChunks * 8192;        // 2 halves x 64 rows x chunks x 64 B
  static constexpr int kPairsPerVStage = kVRawChunks / 2;
  static constexpr int NKS = FP8 ? (kRawRows ? 2 : 3) : 0;   // raw staging depths
  // whole-row key stages also hold the values: the PV MMAs read them there, and a stage is
  // loaded again only once its tile's PV has completed (no value stages); 64 rows keep
  // 1-chunk key stages and 4-chunk value stages
  static constexpr int kValueStages = FP8 && !kRawRows ? 3 : 0;
  // E4M3 q' and P go into the MMAs as hi and lo parts. With whole-row stages each K step
  // is one MMA whose N holds both parts (2 RC columns: S^T and O^T of the hi part and of the
  // lo part, added when read), so that the A operand is read from shared memory once.
  static constexpr int kNC = kRawRows ? 2 * RC : RC;   // tensor-memory columns of S^T / an O^T tile
  static constexpr int kOBase = 2 * kNC;               // first O^T column (after both S^T)
  static_assert(kOBase + 4 * kNC <= 512, "tensor memory budget (S^T and O^T)");
  static constexpr int NVS = kValueStages > 0 ? kValueStages : 1;   // barrier arrays
  static constexpr int kKLoaders = FP8 ? 4 : 1;         // arrivals that fill a K slot
  static constexpr int kVLoaders = 1;
  // FP8: P is computed times 2^kPOffLog2 and written as exact E4M3 hi and lo parts; the
  // reference max moves once a score exceeds it by kRescale (log2 units), so P < 2^8 fits
  static constexpr float kPOffLog2 = FP8 ? 4.f : 0.f;
  static constexpr float kRescale = FP8 ? 4.f : kRescaleLog2;
  static_assert(!FP8 || kKTmemBase + NK * kKTmemSlotCols <= 512, "tensor memory budget");
  static_assert(kSlotsPerTile * KC == 9, "a tile is 9 chunks");
  static constexpr int kDynBytes = 1024 + kQBytes + kNumP * kPBytes + (FP8 ? 0 : NK * kKSlotBytes) +
                                   (FP8 ? 0 : NV * kVSlotBytes) + NKS * kKStageBytes + kValueStages * kVStage;
  static_assert(kDynBytes + kStaticBudget <= kSmemLimit, "shared memory budget");
  static_assert(kNumP * kPBytes >= 8192, "the epilogue's transpose stage");
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

// Two probabilities rounded to bf16 (the bf16 cache's P).
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Walks the key tiles of this CTA's units in the order every role consumes them, with
// per 64-key block h of the current tile the cache row of its first box (rb_h, -1 for a
// block wholly past the sequence end) and the number of its boxes that are loaded (nb_h;
// mla_pages.cuh). A block-table entry outside the pool reads page 0 instead (the combine
// kernel reports it).
struct TileIter {
  int u;
  Unit U;
  int tile;
  int64_t rb0, rb1;
  int nb0, nb1;
  __device__ __forceinline__ uint32_t boxes() const { return (uint32_t)(nb0 + nb1); }
};

// kSub: pages smaller than 64 rows (boxes of a.box_rows rows), else one box per block.
template <bool kSub>
__device__ __forceinline__ void iter_rows(TileIter& it, const DecodeArgs& a) {
  const int32_t* bt = a.block_table + (int64_t)it.U.b * a.MB;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int tok = it.tile * kTileTokens + 64 * h;
    const int64_t r = tok < it.U.L ? page_row(bt, tok, a) : -1;
    const int nb = kSub ? block_boxes(it.U.L - tok, a.box_rows) : (tok < it.U.L ? 1 : 0);
    if (h == 0) { it.rb0 = r; it.nb0 = nb; }
    else { it.rb1 = r; it.nb1 = nb; }
  }
}

// Loads block h of the iterator's tile (chunks from `chunk`): its boxes land at dst,
// dst + box_bytes, ... and complete on `bar`.
template <bool kSub>
__device__ __forceinline__ void load_half(const TileIter& it, const DecodeArgs& a, int h,
                                          const CUtensorMap* map, uint32_t dst, uint32_t bar, int32_t chunk,
                                          uint32_t box_bytes) {
  const int nb = h == 0 ? it.nb0 : it.nb1;
  if (nb == 0) return;
  tma_load_4d(dst, map, bar, 0, 0, chunk, (int32_t)((h == 0 ? it.rb0 : it.rb1) >> 3));
  if (kSub && nb > 1)
    load_more_boxes(kBoxPlain, map, dst, bar, chunk, box_bytes, a.block_table + (int64_t)it.U.b * a.MB, a,
                    it.tile * kTileTokens + 64 * h, nb, 0);
}

template <bool kSub>
__device__ __forceinline__ bool iter_begin(TileIter& it, const DecodeArgs& a, int u0, int u1) {
  it.u = u0;
  if (it.u >= u1) return false;
  it.U = load_unit(a, it.u);
  it.tile = it.U.tb;
  iter_rows<kSub>(it, a);
  return true;
}

template <bool kSub>
__device__ __forceinline__ bool iter_next(TileIter& it, const DecodeArgs& a, int u1) {
  if (++it.tile == it.U.te) {
    if (++it.u >= u1) return false;
    it.U = load_unit(a, it.u);
    it.tile = it.U.tb;
  }
  iter_rows<kSub>(it, a);
  return true;
}

template <int RC, bool FP8, bool kSub>
__global__ void __launch_bounds__(Cfg<RC, FP8>::kThreads, 1)
decode_kernel(const __grid_constant__ DecodeArgs a) {
  using C = Cfg<RC, FP8>;
  constexpr int NK = C::NK, NV = C::NV;
  constexpr int NKS = FP8 ? C::NKS : 1, NVS = FP8 ? C::NVS : 1;
  constexpr int NP = C::kNumP;

  extern __shared__ uint8_t dsmem_raw[];
  __shared__ __align__(8) uint64_t bar_kfull[NK], bar_kempty[NK], bar_vfull[NV], bar_vempty[NV];
  __shared__ __align__(8) uint64_t bar_qfull, bar_qready, bar_qempty;
  __shared__ __align__(8) uint64_t bar_kstage[NKS], bar_ksfree[2 * NKS], bar_vstage[NVS], bar_vsempty[NVS];
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_s_empty[2], bar_p_full[NP], bar_pv[NP];
  __shared__ __align__(8) uint64_t bar_o_empty, bar_drain[2], bar_vaux, bar_never;
  __shared__ uint32_t tmem_base_s;
  __shared__ uint32_t abort_s;
  __shared__ __align__(16) float mref_s[RC];
  __shared__ float alpha_s[RC], tot_s[RC];
  __shared__ int nvis_s[RC];
  __shared__ __align__(16) float qf_s[RC], rowc_s[RC];   // FP8, 16-32 rows: 2^-e of q, score factors
  __shared__ __align__(8) uint64_t bar_qsc, bar_qfree;
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
  const uint32_t sV = sK + (FP8 ? 0 : NK * C::kKSlotBytes);
  const uint32_t sKS = sV + (FP8 ? 0 : NV * kVSlotBytes);
  const uint32_t sVS = sKS + (FP8 ? NKS * C::kKStageBytes : 0);   // raw value stages, C::kVStage each
  uint8_t* gQ = gbase;
  uint8_t* gP = gbase + (sP - sQ);
  uint8_t* gV = gbase + (sV - sQ);
  uint8_t* gKS = gbase + (sKS - sQ);
  uint8_t* gVS = gbase + (sVS - sQ);

  const uint32_t b_kfull = smem_u32(bar_kfull), b_kempty = smem_u32(bar_kempty);
  const uint32_t b_vfull = smem_u32(bar_vfull), b_vempty = smem_u32(bar_vempty);
  const uint32_t b_qfull = smem_u32(&bar_qfull), b_qready = smem_u32(&bar_qready);
  const uint32_t b_qempty = smem_u32(&bar_qempty);
  const uint32_t b_qsc = smem_u32(&bar_qsc), b_qfree = smem_u32(&bar_qfree);
  const uint32_t b_kstage = smem_u32(bar_kstage), b_vstage = smem_u32(bar_vstage);
  // whole-row key stages: half h (keys 64 h ..) of stage s is free again at 2 s + h, once
  // the tile's PV MMAs over those keys have completed
  const uint32_t b_ksfree = smem_u32(bar_ksfree);
  const uint32_t b_vsempty = smem_u32(bar_vsempty);
  const uint32_t b_s_full = smem_u32(bar_s_full), b_s_empty = smem_u32(bar_s_empty);
  const uint32_t b_p_full = smem_u32(bar_p_full), b_pv = smem_u32(bar_pv);
  const uint32_t b_oempty = smem_u32(&bar_o_empty), b_drain = smem_u32(bar_drain);
  const uint32_t b_vaux = smem_u32(&bar_vaux);
  const uint32_t b_never = smem_u32(&bar_never);   // tests: a barrier nothing arrives on
  volatile uint32_t* abort_flag = &abort_s;
  uint32_t* err = a.err;
  const uint32_t box_rows = kSub ? (uint32_t)a.box_rows : 64u;   // rows of one key/value box

  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(b_kfull + 8 * i, C::kKLoaders);
      mbar_init(b_kempty + 8 * i, 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(b_vfull + 8 * i, C::kVLoaders);
      mbar_init(b_vempty + 8 * i, 1);
    }
    mbar_init(b_qfull, 1);
    mbar_init(b_qready, 4);
    for (int i = 0; i < NKS; ++i) {
      mbar_init(b_kstage + 8 * i, 1);
      mbar_init(b_ksfree + 8 * (2 * i), 1);
      mbar_init(b_ksfree + 8 * (2 * i + 1), 1);
    }
    for (int i = 0; i < NVS; ++i) {
      mbar_init(b_vstage + 8 * i, 1);
      mbar_init(b_vsempty + 8 * i, 1);
    }
    mbar_init(b_qempty, 1);
    mbar_init(b_qsc, 1);     // FP8, 16-32 rows: the Q converters, with the row factors
    mbar_init(b_qfree, 1);   // the softmax warps, once they have read them
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
    mbar_init(b_drain + 8, 1);
    mbar_init(b_vaux, 1);
    mbar_init(b_never, 1);
    abort_s = 0u;
    fence_mbarrier_init();
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  // the set-up above overlaps the scheduler (programmatic dependent launch); its output is
  // read only after it has completed
  griddep_wait();

  // this CTA's units: a contiguous range of the scheduler's list
  const int u0 = a.cta_first[blockIdx.x], u1 = a.cta_first[blockIdx.x + 1];
  const int R = a.R;

  auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
    return mbar_wait(bar, parity, abort_flag, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
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
  if (!FP8 && warp == 0) {
    // ============================================================ key producer (bf16)
    // One thread: every key slot of every tile is two TMA boxes (one per 64-row page
    // half) of KC chunks; a half wholly past the sequence end is not loaded (its scores
    // are masked).
    if (lane == 0) {
      TileIter it;
      bool more = iter_begin<kSub>(it, a, u0, u1);
      bool ok = true;
      uint32_t p = 0;
      const uint32_t box_bytes = (C::kKSlotBytes / 128) * box_rows;
      while (more && ok) {
        for (int sl = 0; sl < C::kSlotsPerTile; ++sl, ++p) {
          const uint32_t slot = p % NK;
          ok = wait(b_kempty + 8 * slot, ((p / NK) & 1) ^ 1);
          if (!ok) break;
          const uint32_t bar = b_kfull + 8 * slot, dst = sK + slot * C::kKSlotBytes;
          mbar_arrive_expect_tx(bar, it.boxes() * box_bytes);
          for (int h = 0; h < 2; ++h)
            load_half<kSub>(it, a, h, &a.tm_k, dst + h * (C::kKSlotBytes / 2), bar, sl * C::KC, box_bytes);
        }
        if (ok) more = iter_next<kSub>(it, a, u1);
      }
      // the last loads issued have landed before the CTA may exit
      volatile uint32_t no_abort = 0;
      for (uint32_t q = p > (uint32_t)NK ? p - NK : 0; q < p; ++q)
        mbar_wait(b_kfull + 8 * (q % NK), (q / NK) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    }
  } else if (!FP8 && warp == 2) {
    // ============================================================ value producer (bf16)
    // Every value chunk pair: two TMA boxes (re-read from L2, so that no slot lives from
    // QK^T to PV). On the last tile of a unit the rows from the sequence end up to the end
    // of the last 16-key MMA step are overwritten with zeros (the cache may hold NaN there
    // and 0 * NaN is NaN inside the MMA); rows past that step are never read.
    TileIter it;
    bool more = iter_begin<kSub>(it, a, u0, u1);
    bool ok = true;
    uint32_t p = 0, aux = 0;
    const uint32_t box_bytes = (kVSlotBytes / 128) * box_rows;
    while (more && ok) {
      const int valid = it.U.L - it.tile * kTileTokens;
      const bool tail = valid < kTileTokens;
      for (int j = 0; j < kPairsPerTile; ++j, ++p) {
        const uint32_t slot = p % NV;
        ok = wait_warp(b_vempty + 8 * slot, ((p / NV) & 1) ^ 1);
        if (!ok) break;
        const uint32_t dst = sV + slot * kVSlotBytes;
        const uint32_t bar = tail ? b_vaux : b_vfull + 8 * slot;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar, it.boxes() * box_bytes);
          for (int h = 0; h < 2; ++h)
            load_half<kSub>(it, a, h, &a.tm_v, dst + h * (kVSlotBytes / 2), bar, 2 * j, box_bytes);
        }
        if (tail) {
          ok = wait_warp(b_vaux, aux & 1);
          ++aux;
          if (!ok) break;
          const int nrow = min(kTileTokens, (valid + 15) & ~15) - valid;   // 0..15 rows
          uint8_t* g = gV + slot * kVSlotBytes;
          for (int idx = lane; idx < nrow * 16; idx += 32) {   // per row: 2 chunks x 8 units
            const int row = valid + (idx >> 4), c = (idx >> 3) & 1, u16 = idx & 7;
            *reinterpret_cast<uint4*>(g + (row >> 3) * 2048 + c * 1024 + (row & 7) * 128 + u16 * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_vfull + 8 * slot);
        }
      }
      if (ok) more = iter_next<kSub>(it, a, u1);
    }
    if (lane == 0) {
      volatile uint32_t no_abort = 0;
      for (uint32_t q = p > (uint32_t)NV ? p - NV : 0; q < p; ++q)
        mbar_wait(b_vfull + 8 * (q % NV), (q / NV) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ============================================================ QK^T issuer
    // One thread, in program order: per unit the Q load (TMA), per tile the S^T buffer,
    // then every key slot: wait full, 4*KC MMAs, release the slot when they complete.
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(128, RC, FP8 ? 0u : 1u, 0, 0);
      // descriptors built once, advanced by constants (the start field counts 16 B units)
      const uint64_t dK0 = make_sdesc(sK, 16, C::kKGroupStride, kSwizzle128);
      const uint64_t dQ0 = make_sdesc(sQ, 16, 1024, kSwizzle128);
      const uint64_t dKS = make_sdesc(sKS, 16, 9 * 512, kSwizzle64);
      const uint64_t dQ8 = make_sdesc(sQ, 16, 512, kSwizzle64);
      const uint32_t idesc_qk8 = make_idesc(128, 2 * RC, 0, 0, 0);
      uint32_t n = 0, kp = 0, uc = 0;
      bool ok = true;
      for (int u = u0; u < u1 && ok; ++u, ++uc) {
        const Unit U = load_unit(a, u);
        // Q of the unit, once the previous unit's QK^T MMAs have released the buffer
        ok = wait(b_qempty, (uc & 1) ^ 1);
        if (!ok) break;
        mbar_arrive_expect_tx(b_qfull, 9 * RC * 128);
        for (int c = 0; c < 9; ++c) tma_load_3d(sQ + c * RC * 128, &a.tm_q, b_qfull, c * 64, U.g * RC, U.b);
        ok = wait(FP8 ? b_qready : b_qfull, uc & 1);
        for (int k = 0; k < U.te - U.tb && ok; ++k, ++n) {
          ok = wait(b_s_empty + 8 * (n & 1), ((n >> 1) & 1) ^ 1);
          const uint32_t d = tmem + (n & 1) * C::kNC;
          if constexpr (C::kRawRows) {
            // E4M3 keys straight from the tile's whole-row stage (K-major, 64-byte swizzle,
            // 8-row groups 4.5 KB apart) against q' = q 2^e as E4M3 hi and lo (K-major, each
            // 1 KB block of 8 rows x 64 columns: hi in its first 512 B, lo in its second)
            const uint32_t st = n % NKS;
            ok = ok && wait(b_kstage + 8 * st, (n / NKS) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint64_t as = dKS + (uint64_t)(st * (C::kKStageBytes >> 4));
            // N = 2 RC: the 512-byte groups of 8 rows alternate hi and lo, so that S^T column
            // 16 g + i is row 8 g + i of K . hi and column 16 g + 8 + i the same row of K . lo
#pragma unroll
            for (int c = 0; c < 9; ++c) {
              const uint64_t bd = dQ8 + (uint64_t)(c * (RC * 128 >> 4));
#pragma unroll
              for (int kk = 0; kk < 2; ++kk)
                umma_f8(d, as + (uint64_t)(c * (512 >> 4) + 2 * kk), bd + 2 * kk, idesc_qk8, (c | kk) != 0);
            }
          }
          for (int sl = 0; !C::kRawRows && sl < C::kSlotsPerTile && ok; ++sl, ++kp) {
            const uint32_t ks = kp % NK;
            ok = wait(b_kfull + 8 * ks, (kp / NK) & 1);
            if (!ok) break;
            tc_fence_after();
            if (FP8) {
              // keys dequantised into tensor memory: 8 columns per K = 16 step
              const uint32_t at0 = tmem + C::kKTmemBase + ks * C::kKTmemSlotCols;
#pragma unroll
              for (int cc = 0; cc < C::KC; ++cc) {
                const int c = sl * C::KC + cc;
                const uint64_t bd = dQ0 + (uint64_t)(c * (RC * 128 >> 4));
                const uint32_t at = at0 + cc * 32;
                umma_f16_ts(d, at, bd, idesc_qk, c != 0);
                umma_f16_ts(d, at + 8, bd + 2, idesc_qk, 1);
                umma_f16_ts(d, at + 16, bd + 4, idesc_qk, 1);
                umma_f16_ts(d, at + 24, bd + 6, idesc_qk, 1);
              }
            } else {
              const uint64_t ad0 = dK0 + (uint64_t)(ks * (C::kKSlotBytes >> 4));
#pragma unroll
              for (int cc = 0; cc < C::KC; ++cc) {
                const int c = sl * C::KC + cc;
                const uint64_t ad = ad0 + (uint64_t)(cc * (C::kKChunkStride >> 4));
                const uint64_t bd = dQ0 + (uint64_t)(c * (RC * 128 >> 4));
                umma_f16(d, ad, bd, idesc_qk, c != 0);
                umma_f16(d, ad + 2, bd + 2, idesc_qk, 1);
                umma_f16(d, ad + 4, bd + 4, idesc_qk, 1);
                umma_f16(d, ad + 6, bd + 6, idesc_qk, 1);
              }
            }
            umma_commit(b_kempty + 8 * ks);
          }
          if (ok) umma_commit(b_s_full + 8 * (n & 1));
        }
        if (ok) umma_commit(b_qempty);
      }
      // drain: every MMA issued has completed before tensor memory is released
      umma_commit(b_drain);
      volatile uint32_t no_abort = 0;
      mbar_wait(b_drain, 0, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    }
  } else if (warp == C::kPvWarp) {
    // ============================================================ PV issuer
    // One thread, in program order: per tile the softmax's P^T (and, for the first tile of
    // a unit, the epilogue's release of O^T), then every value chunk pair: wait full,
    // 8 MMAs (fewer on a partial last tile), release the slot when they complete. FP8: the
    // MMAs read the raw E4M3 value stages as they landed (kind::f8f6f4, K = 32), each K
    // step once with P's hi part and once with its lo part.
    if (lane == 0) {
      const uint32_t idesc_pv = make_idesc(128, RC, FP8 ? 0u : 1u, 1, 1);
      const uint64_t dV0 = make_sdesc(sV, C::kVChunkStride, C::kVGroupStride, kSwizzle128);
      const uint64_t dP0 = make_sdesc(sP, 8 * C::kPRow, 8 * C::kPRow, C::kPSwz);
      // FP8 raw value stage [2 halves][8 groups][VC chunks][8 rows][64 B]: MN-major, chunks
      // 512 B apart (leading offset), 8-key groups VC x 512 B apart. P^T hi (then lo, 128 RC
      // bytes on): [8-key group][RC / 16 cores][8 keys][16 B], MN-major without swizzle, where
      // the leading offset steps along K (8-key groups, 8 RC bytes) and the stride offset
      // along MN (16-byte cores, 128 B).
      constexpr uint32_t kVC = C::kVRawChunks;
      const uint64_t dVS0 = make_sdesc(sVS, 512, kVC * 512, kSwizzle64);
      const uint64_t dP8 = make_sdesc(sP, 8 * RC, 128, kSwizzleNone);
      const uint64_t dKS0 = make_sdesc(sKS, 512, 9 * 512, kSwizzle64);   // whole-row key stages
      // whole-row stages: P^T [8-key group][2 RC / 16 cores: hi, then lo][8 keys][16 B]
      const uint64_t dP8s = make_sdesc(sP, 16 * RC, 128, kSwizzleNone);
      const uint32_t idesc_pv8 = make_idesc(128, 2 * RC, 0, 1, 1);
      uint32_t n = 0, vp = 0, uc = 0;
      bool ok = true;
      for (int u = u0; u < u1 && ok; ++u, ++uc) {
        const Unit U = load_unit(a, u);
        for (int k = 0; k < U.te - U.tb && ok; ++k, ++n) {
          const uint32_t pb = n % NP;
          ok = wait(b_p_full + 8 * pb, (n / NP) & 1);
          if (ok && k == 0) ok = wait(b_oempty, (uc & 1) ^ 1);
          const int valid = U.L - (U.tb + k) * kTileTokens;
          if constexpr (FP8 && C::kRawRows) {
            // the values are the first 8 chunks of the tile's whole-row key stage
            // ([2 halves][8 groups][9 chunks][8 rows][64 B]); each half is released once the
            // MMAs of its two K steps complete (its keys' QK^T completed before P was ready)
            const int ksteps = valid >= kTileTokens ? 4 : (valid + 31) / 32;
            const uint32_t st = n % NKS;
            ok = wait(b_kstage + 8 * st, (n / NKS) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint64_t as = dKS0 + (uint64_t)(st * (C::kKStageBytes >> 4));
            // N = 2 RC: P^T's cores hold hi (O^T columns 0 .. RC - 1) then lo (RC .. 2 RC - 1)
            const uint64_t bs = dP8s + (uint64_t)(pb * (C::kPBytes >> 4));
            // consecutive MMAs go to the four O^T tiles in turn (independent accumulators)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (kk >= ksteps) break;
#pragma unroll
              for (int j = 0; j < kPairsPerTile; ++j)
                umma_f8(tmem + C::kOBase + j * C::kNC, as + (uint64_t)((2 * j * 512 + kk * 4 * 9 * 512) >> 4),
                        bs + (uint64_t)((kk * 64 * RC) >> 4), idesc_pv8, !(k == 0 && kk == 0));
              if (kk == 1) umma_commit(b_ksfree + 8 * (2 * st));
            }
            if (ksteps < 2) umma_commit(b_ksfree + 8 * (2 * st));
            umma_commit(b_ksfree + 8 * (2 * st + 1));
          } else if constexpr (FP8) {
            const int ksteps = valid >= kTileTokens ? 4 : (valid + 31) / 32;
            const uint64_t bh = dP8 + (uint64_t)(pb * (C::kPBytes >> 4));
            for (int j0 = 0; j0 < kPairsPerTile && ok; j0 += C::kPairsPerVStage, ++vp) {
              const uint32_t st = vp % NVS;
              ok = wait(b_vstage + 8 * st, (vp / NVS) & 1);
              if (!ok) break;
              tc_fence_after();
              const uint64_t as = dVS0 + (uint64_t)(st * (C::kVStage >> 4));
              for (int pin = 0; pin < C::kPairsPerVStage; ++pin) {
                const uint32_t d = tmem + (2 + j0 + pin) * RC;
                for (int kk = 0; kk < ksteps; ++kk) {
                  const uint64_t ad = as + (uint64_t)((2 * pin * 512 + kk * 4 * kVC * 512) >> 4);
                  const uint64_t bd = bh + (uint64_t)((kk * 32 * RC) >> 4);
                  umma_f8(d, ad, bd, idesc_pv, !(k == 0 && kk == 0));        // V . P hi
                  umma_f8(d, ad, bd + (uint64_t)((128 * RC) >> 4), idesc_pv, 1u);   // V . P lo
                }
              }
              umma_commit(b_vsempty + 8 * st);
            }
          } else {
            const int ksteps = valid >= kTileTokens ? 8 : (valid + 15) / 16;
            const uint64_t bd0 = dP0 + (uint64_t)(pb * (C::kPBytes >> 4));
            for (int j = 0; j < kPairsPerTile && ok; ++j, ++vp) {
              const uint32_t vs = vp % NV;
              ok = wait(b_vfull + 8 * vs, (vp / NV) & 1);
              if (!ok) break;
              tc_fence_after();
              const uint64_t ad0 = dV0 + (uint64_t)(vs * (kVSlotBytes >> 4));
              const uint32_t d = tmem + (2 + j) * RC;
              if (ksteps == 8) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  umma_f16(d, ad0 + kk * (2 * C::kVGroupStride >> 4), bd0 + kk * (16 * C::kPRow >> 4), idesc_pv,
                           !(k == 0 && kk == 0));
              } else {
                for (int kk = 0; kk < ksteps; ++kk)
                  umma_f16(d, ad0 + kk * (2 * C::kVGroupStride >> 4), bd0 + kk * (16 * C::kPRow >> 4), idesc_pv,
                           !(k == 0 && kk == 0));
              }
              umma_commit(b_vempty + 8 * vs);
            }
          }
          if (ok) umma_commit(b_pv + 8 * pb);
        }
      }
      umma_commit(b_drain + 8);
      volatile uint32_t no_abort = 0;
      mbar_wait(b_drain + 8, 0, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    }
  } else if (warp >= 4 && warp < 8) {
    // ============================================================ softmax / epilogue
    const int w4 = warp - 4;
    const int t = w4 * 32 + lane;                       // key within the tile = TMEM lane
    const uint32_t lane_addr = (uint32_t)(w4 * 32) << 16;
    const float kvs = FP8 ? __ldg(a.kv_scale) : 1.0f;
    const float c_log2 = a.softmax_scale * kvs * kLog2e;
    const float kvo = kvs;                              // value scale (FP8: kv_scale)
    uint32_t gn = 0;
    bool ok = true;
    float lsum[RC];
    for (int u = u0; u < u1 && ok; ++u) {
      const Unit U = load_unit(a, u);
      const int T = U.te - U.tb;
      const int row0 = U.g * RC;
      // keys visible to row r: L - s_q + 1 + i(r) when causal (i = the row's new-token
      // index), else L; only tiles that reach past L - s_q + 1 (or L) need the mask
      if (t < RC) {
        mref_s[t] = -INFINITY;
        nvis_s[t] = a.causal ? min(U.L, U.L - a.s_q + 1 + (row0 + t) / a.H) : U.L;
      }
      const int mask_from = a.causal ? U.L - a.s_q + 1 : U.L;
      if constexpr (C::kRawRows) {
        // the unit's score factors: softmax scale x log2 e x 2^-e of the row's q
        ok = wait_softmax(b_qsc, (uint32_t)(u - u0) & 1);
        if (!ok) break;
        if (t < RC) rowc_s[t] = c_log2 * qf_s[t];
        named_bar_sync(kSoftmaxBar, 128);
        if (t == 0) mbar_arrive(b_qfree);
      }
#pragma unroll
      for (int r = 0; r < RC; ++r) lsum[r] = 0.f;
      named_bar_sync(kSoftmaxBar, 128);
      for (int k = 0; k < T && ok; ++k) {
        const uint32_t n = gn + k, sb = n & 1, pb = n % NP;
        if (a.test_stall && n == 0) {
          ok = wait_softmax(b_never, 0);            // tests: this wait runs out
          if (!ok) break;
        }
        ok = wait_softmax(b_s_full + 8 * sb, (n >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        float s[RC];
        if constexpr (C::kRawRows) {
          // columns 16 g .. 16 g + 7: rows 8 g .. of K . hi; the next 8: the same rows of K . lo
#pragma unroll
          for (int g = 0; g < RC / 8; g += 2) {
            float v[2][16];
            tmem_ld16(tmem + lane_addr + sb * C::kNC + 16 * g, v[0]);
            tmem_ld16(tmem + lane_addr + sb * C::kNC + 16 * g + 16, v[1]);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int i = 0; i < 8; ++i) s[8 * (g + h) + i] = v[h][i] + v[h][8 + i];
          }
        } else {
#pragma unroll
          for (int c = 0; c < RC / 16; ++c) tmem_ld16(tmem + lane_addr + sb * RC + 16 * c, s + 16 * c);
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(b_s_empty + 8 * sb);

        const int j = (U.tb + k) * kTileTokens + t;
        // the reference maxima are read from shared memory (a broadcast) where they are
        // used, rather than held in RC registers
        auto mref4 = [&](int r) { return *reinterpret_cast<const float4*>(mref_s + r); };
        // the score factor of 4 rows: one constant, or (E4M3 q') per row
        auto factors = [&](int r, float* cc) {
          if constexpr (C::kRawRows) {
            const float4 c4 = *reinterpret_cast<const float4*>(rowc_s + r);
            cc[0] = c4.x; cc[1] = c4.y; cc[2] = c4.z; cc[3] = c4.w;
          } else {
            cc[0] = cc[1] = cc[2] = cc[3] = c_log2;
          }
        };
        bool need = false;
        if ((U.tb + k + 1) * kTileTokens <= mask_from) {
#pragma unroll
          for (int r = 0; r < RC; r += 4) {
            const float4 m4 = mref4(r);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
            float cc[4];
            factors(r, cc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              s[r + i] *= cc[i];
              need |= s[r + i] > mm[i] + C::kRescale;
            }
          }
        } else {
#pragma unroll
          for (int r = 0; r < RC; r += 4) {
            const float4 m4 = mref4(r);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
            float cc[4];
            factors(r, cc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              s[r + i] = j < nvis_s[r + i] ? s[r + i] * cc[i] : -INFINITY;
              need |= s[r + i] > mm[i] + C::kRescale;
            }
          }
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
        // P^T row of this key, in registers until its buffer is free. bf16: RC / 2 words of
        // pairs. FP8: P times 2^4 as E4M3 hi bytes (words 0 .. RC / 4 - 1) and lo bytes
        // (the rest), four rows per word.
        uint32_t pw[RC / 2];
#pragma unroll
        for (int r = 0; r < RC; r += 4) {
          const float4 m4 = mref4(r);
          const float mm[4] = {m4.x - C::kPOffLog2, m4.y - C::kPOffLog2, m4.z - C::kPOffLog2, m4.w - C::kPOffLog2};
          float pr[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pr[i] = s[r + i] == -INFINITY ? 0.f : ex2_approx(s[r + i] - mm[i]);
            lsum[r + i] += pr[i];   // the normaliser sums the unrounded probabilities
          }
          if constexpr (FP8) {
            const uint32_t o0 = split_e4m3x2(pr[0], pr[1]), o1 = split_e4m3x2(pr[2], pr[3]);
            pw[r / 4] = __byte_perm(o0, o1, 0x5410);
            pw[RC / 4 + r / 4] = __byte_perm(o0, o1, 0x7632);
          } else {
            pw[r / 2] = pack2_bf16(pr[0], pr[1]);
            pw[r / 2 + 1] = pack2_bf16(pr[2], pr[3]);
          }
        }
        // the buffer's previous user, PV(n - NP), must have completed
        if (n >= (uint32_t)NP) {
          ok = wait_softmax(b_pv + 8 * pb, ((n / NP) - 1) & 1);
          if (!ok) break;
        }
        uint8_t* prow = gP + pb * C::kPBytes;
        if constexpr (C::kRawRows) {
          // [8-key group][2 RC / 16 cores: hi, then lo][8 keys][16 B]
#pragma unroll
          for (int c = 0; c < RC / 8; ++c) {
            uint8_t* q = prow + (t >> 3) * (16 * RC) + c * 128 + (t & 7) * 16;
            *reinterpret_cast<uint4*>(q) = make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
          }
        } else if constexpr (FP8) {
          // [8-key group][RC / 16 cores][8 keys][16 B] for hi, the same for lo 128 RC bytes on
#pragma unroll
          for (int c = 0; c < RC / 16; ++c) {
            uint8_t* q = prow + (t >> 3) * (8 * RC) + c * 128 + (t & 7) * 16;
            *reinterpret_cast<uint4*>(q) = make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
            *reinterpret_cast<uint4*>(q + 128 * RC) =
                make_uint4(pw[RC / 4 + 4 * c], pw[RC / 4 + 4 * c + 1], pw[RC / 4 + 4 * c + 2], pw[RC / 4 + 4 * c + 3]);
          }
        } else {
#pragma unroll
          for (int u16 = 0; u16 < C::kPRow / 16; ++u16)
            *reinterpret_cast<uint4*>(prow + p_offset<C::kPRow>(t, u16)) =
                make_uint4(pw[4 * u16], pw[4 * u16 + 1], pw[4 * u16 + 2], pw[4 * u16 + 3]);
        }
        fence_proxy_async_smem();
        if (rescale) {
          // O^T holds tiles up to k-1 of this unit: wait for PV(n-1), then scale in place
          ok = wait_softmax(b_pv + 8 * ((n - 1) % NP), ((n - 1) / NP) & 1);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int jt = 0; jt < 4; ++jt) {
            // whole-row stages: columns c >= RC / 16 hold the lo part of rows 16 c - RC ..
#pragma unroll
            for (int c = 0; c < C::kNC / 16; ++c) {
              float o[16];
              const uint32_t ta = tmem + lane_addr + C::kOBase + jt * C::kNC + 16 * c;
              tmem_ld16(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= alpha_s[(16 * c + i) % RC];
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
      if (t < RC) {
        const float tot = (wmax_s[t] + wmax_s[RC + t]) + (wmax_s[2 * RC + t] + wmax_s[3 * RC + t]);
        tot_s[t] = tot;
        alpha_s[t] = tot > 0.f ? kvo / tot : 0.f;     // the row's output factor
      }
      named_bar_sync(kSoftmaxBar, 128);
      const bool direct = U.slot < 0;
      // Each warp holds output columns 128 jt + 32 w4 + lane (its TMEM lanes) of 16 rows
      // per load. It transposes them through 2 KB of the (now idle) P^T buffers, 16-byte
      // blocks XOR-swizzled by row, so that each lane stores 16 consecutive columns of one
      // row: 16-byte vector stores instead of one 2-byte store per row.
      float* stage = reinterpret_cast<float*>(gP) + w4 * 512;
      const int si = lane >> 1, sh = lane & 1;
#pragma unroll 1
      for (int jt = 0; jt < 4; ++jt) {
#pragma unroll 1
        for (int c = 0; c < RC / 16; ++c) {
          float o[16];
          tmem_ld16(tmem + lane_addr + C::kOBase + jt * C::kNC + 16 * c, o);
          if constexpr (C::kRawRows) {
            // plus the lo part's columns RC + 16 c ..
            float o2[16];
            tmem_ld16(tmem + lane_addr + C::kOBase + jt * C::kNC + RC + 16 * c, o2);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] += o2[i];
          }
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            stage[i * 32 + ((((lane >> 2) ^ (i & 7)) << 2) | (lane & 3))] = o[i] * alpha_s[16 * c + i];
          __syncwarp();
          float v[16];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 x = *reinterpret_cast<const float4*>(stage + si * 32 + (((4 * sh + m) ^ (si & 7)) << 2));
            v[4 * m] = x.x;
            v[4 * m + 1] = x.y;
            v[4 * m + 2] = x.z;
            v[4 * m + 3] = x.w;
          }
          __syncwarp();
          const int r = 16 * c + si, rg = row0 + r;
          const int col = 128 * jt + 32 * w4 + 16 * sh;
          if (rg < R) {
            if (direct) {
              uint32_t w[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
                w[k] = *reinterpret_cast<uint32_t*>(&h);
              }
              uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)U.b * R + rg) * kDV + col);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
              float4* dst = reinterpret_cast<float4*>(a.part_o + ((int64_t)U.slot * RC + r) * kDV + col);
#pragma unroll
              for (int m = 0; m < 4; ++m) dst[m] = make_float4(v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]);
            }
          }
        }
      }
      if (t < RC && row0 + t < R) {
        const float tot = tot_s[t];
        // FP8: P was computed times 2^kPOffLog2, and so was the row sum
        const float l = tot > 0.f ? (mref_s[t] + __log2f(tot) - C::kPOffLog2) * kLn2 : -INFINITY;
        if (direct) a.lse[(int64_t)U.b * R + row0 + t] = l;
        else a.part_lse[(int64_t)U.slot * RC + t] = l;
      }
      tc_fence_before();
      mbar_arrive(b_oempty);
      named_bar_sync(kSoftmaxBar, 128);
      gn += T;
    }
  } else if (FP8 && C::kRawRows && warp >= 8) {
    // ============================================================ FP8 Q converters (16-32 rows)
    // Each unit's RC query rows, bf16 as TMA landed them ([9 chunks][RC rows][128 B], 128-byte
    // swizzle), become q' = q 2^e (the row's largest |q| in [128, 256)) written as E4M3 hi
    // and lo in place: every 1 KB block of 8 rows x 64 columns becomes hi in its first 512
    // bytes and lo in its second (8 rows x 64 bytes, 64-byte swizzled each), the QK^T MMAs'
    // B operand. hi + lo is q' exactly (8 significant bits). A warp owns whole 8-row groups,
    // so its reads of a block precede its writes there; lane 4 q + p holds 16-byte units p
    // and p + 4 of row q of each block. The row factors 2^-e go to qf_s for the softmax.
    const int qrow = lane >> 2, part = lane & 3;
    uint32_t uq = 0;
    for (int u = u0; u < u1; ++u, ++uq) {
      const bool mine = threadIdx.x != 256 || (wait(b_qfull, uq & 1) && (uq == 0 || wait(b_qfree, (uq - 1) & 1)));
      if (named_bar_or(kKeyDqBar, kKeyDqThreads, !mine)) break;
      for (int g = warp - 8; g < RC / 8; g += 4) {
        auto block_of = [&](int c) -> uint8_t* { return gQ + c * (RC * 128) + g * 1024; };
        // pass 1: the row's largest |q| (this lane's 18 units, then the row's 4 lanes)
        __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll
        for (int c = 0; c < 9; ++c)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 v = *reinterpret_cast<const uint4*>(block_of(c) + qrow * 128 + (((part + 4 * h) ^ qrow) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[k])));
          }
        float mx = fmaxf(__low2float(m2), __high2float(m2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // e = 7 - floor(log2 max|q|), so that the row's largest |q'| lies in [128, 256)
        int e = 0;
        if (mx > 0.f) e = min(max(7 - ((int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127), -126), 126);
        const float f = __uint_as_float((uint32_t)(e + 127) << 23);
        // pass 2, block by block: the warp's reads of a block precede its writes there
#pragma unroll 3
        for (int c = 0; c < 9; ++c) {
          uint8_t* blk = block_of(c);
          uint4 v[2];
#pragma unroll
          for (int h = 0; h < 2; ++h)
            v[h] = *reinterpret_cast<const uint4*>(blk + qrow * 128 + (((part + 4 * h) ^ qrow) << 4));
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int un = part + 4 * h;           // columns 8 un .. 8 un + 7 of the block
            const uint32_t w[4] = {v[h].x, v[h].y, v[h].z, v[h].w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              o[k] = split_e4m3x2(__uint_as_float(w[k] << 16) * f, __uint_as_float(w[k] & 0xFFFF0000u) * f);
            // 8 bytes: half (un % 2) of the 16-byte unit un / 2 of the 64-byte row
            const uint32_t off = qrow * 64 + (((un >> 1) ^ ((qrow >> 1) & 3)) << 4) + (un & 1) * 8;
            *reinterpret_cast<uint2*>(blk + off) = make_uint2(__byte_perm(o[0], o[1], 0x5410), __byte_perm(o[2], o[3], 0x5410));
            *reinterpret_cast<uint2*>(blk + 512 + off) =
                make_uint2(__byte_perm(o[0], o[1], 0x7632), __byte_perm(o[2], o[3], 0x7632));
          }
        }
        if (part == 0) qf_s[8 * g + qrow] = __uint_as_float((uint32_t)(127 - e) << 23);
      }
      fence_proxy_async_smem();
      named_bar_sync(kKeyDqBar, kKeyDqThreads);
      if (threadIdx.x == 256) mbar_arrive(b_qsc);
      if (lane == 0) mbar_arrive(b_qready);
    }
  } else if (FP8 && warp >= 8) {
    // ============================================================ FP8 keys (+ Q)
    // Warps 8-11, one thread per key row of the tile (thread gi = tensor-memory lane gi).
    // Every key position (KC chunks) is converted from its raw staging slot into a
    // tensor-memory key slot, which the QK^T MMAs read as their A operand (E4M3 -> fp16 is
    // exact; key rows past the sequence end are masked by the softmax). At the start of
    // each unit the group converts that unit's Q from bf16 to fp16 in place.
    // Thread 0 does the waits (the group barrier passes them on), then refills the raw
    // staging slots the group has just finished reading, with TMA boxes (one per 64-row
    // page half).
    const int gi = threadIdx.x - 256;                   // 0..127 = key row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp & 3) << 21);   // (32 * (warp % 4)) << 16
    TileIter kc, ki;                                    // consume / issue cursors
    bool kmore = iter_begin<kSub>(kc, a, u0, u1);
    // whole-row stages are loaded by warp 2 (they are released by the PV MMAs)
    bool kimore = !C::kRawRows && gi == 0 && iter_begin<kSub>(ki, a, u0, u1);
    // raw stages: kip issued, kfreed read by every thread (free again), kwaited landed
    int kic = 0;
    uint32_t kip = 0, kcp = 0, uq = 0, kfreed = 0, kwaited = 0;
    auto top_up = [&]() {
      while (kimore && kip < kfreed + NKS) {
        const uint32_t sl = kip % NKS, bar = b_kstage + 8 * sl, dst = sKS + sl * C::kKStageBytes;
        const uint32_t box_bytes = (C::kKStageBytes / 128) * box_rows;
        // a whole-row stage (all 9 chunks) or the KC chunks of one position
        const int32_t c0 = C::kRawRows ? 0 : kic * C::KC;
        mbar_arrive_expect_tx(bar, ki.boxes() * box_bytes);
        for (int h = 0; h < 2; ++h)
          load_half<kSub>(ki, a, h, &a.tm_k, dst + h * (C::kKStageBytes / 2), bar, c0, box_bytes);
        if (C::kRawRows || ++kic == C::kSlotsPerTile) { kic = 0; kimore = iter_next<kSub>(ki, a, u1); }
        ++kip;
      }
    };
    if (gi == 0) top_up();
    // staging row gi of a key stage: half gi/64, group (gi/8)%8, row gi%8; each 64-byte
    // chunk row's four 16-byte units are 64-byte swizzled by row (the key map's swizzle)
    const int kr7 = gi & 7;
    const uint32_t krow_off =
        (uint32_t)(gi >> 6) * (C::kKStageBytes / 2) + ((gi >> 3) & 7) * (C::kKRawChunks * 512) + kr7 * 64;
    bool ok = true;
    while (kmore && ok) {
      if (kc.tile == kc.U.tb) {
        // ---- Q of the unit, bf16 -> fp16 in place, once the QK^T issuer has loaded it
        const bool mine = gi != 0 || wait(b_qfull, uq & 1);
        ok = !named_bar_or(kKeyDqBar, kKeyDqThreads, !mine);
        if (!ok) break;
        bool q_bad = false;
        for (int i = gi; i < C::kQBytes / 16; i += kKeyDqThreads) {
          uint4* qp = reinterpret_cast<uint4*>(gQ + 16 * i);
          const uint4 v = *qp;
          uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
            q_bad |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
            __half2 h = __floats2half2_rn(lo, hi);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
          }
          *qp = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (q_bad) atomicOr(err, MLA_DEVERR_Q_RANGE);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_qready);
        ++uq;
      }
      for (int sl = 0; sl < C::kSlotsPerTile && ok; ++sl) {
        // position kcp reads raw stage rs (waited for at the stage's first position)
        const uint32_t rs = kcp / C::kKPosPerStage, st = rs % NKS, ks = kcp % NK;
        const int pin = (int)(kcp % C::kKPosPerStage);
        const bool mine = gi != 0 || ((pin != 0 || wait(b_kstage + 8 * st, (rs / NKS) & 1)) &&
                                      wait(b_kempty + 8 * ks, ((kcp / NK) & 1) ^ 1));
        ok = !named_bar_or(kKeyDqBar, kKeyDqThreads, !mine);   // everyone is done with the last position
        if (!ok) break;
        if (pin == 0) kwaited = rs + 1;
        if (C::kKPosPerStage == 1) {
          kfreed = kcp;                                  // the previous position's stage
          if (gi == 0) top_up();
        }
        tc_fence_after();
        const uint8_t* src = gKS + st * C::kKStageBytes + krow_off + pin * (C::KC * 512);
        const uint32_t tbase = lane_base + C::kKTmemBase + ks * C::kKTmemSlotCols;
        // one chunk per iteration: the five roles of a CTA share the SM's instruction
        // caches, and the fully unrolled position (KC chunks) lost more to instruction
        // fetch stalls than the loop costs (measured 10% slower with 16 query rows)
#pragma unroll 1
        for (int cc = 0; cc < C::KC; ++cc) {
          uint4 raw[4];
#pragma unroll
          for (int u16 = 0; u16 < 4; ++u16)
            raw[u16] = *reinterpret_cast<const uint4*>(src + cc * 512 + ((u16 ^ ((kr7 >> 1) & 3)) << 4));
          uint32_t w[32];
#pragma unroll
          for (int u16 = 0; u16 < 4; ++u16) {
            const uint32_t b4[4] = {raw[u16].x, raw[u16].y, raw[u16].z, raw[u16].w};
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              w[8 * u16 + 2 * k2] = e4m3x2_to_f16x2(b4[k2] & 0xFFFFu);
              w[8 * u16 + 2 * k2 + 1] = e4m3x2_to_f16x2(b4[k2] >> 16);
            }
          }
          tmem_st16u(tbase + cc * 32, w);
          tmem_st16u(tbase + cc * 32 + 16, w + 16);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_kfull + 8 * ks);
        ++kcp;
        if (C::kKPosPerStage > 1 && pin == C::kKPosPerStage - 1) {
          // every thread has read the stage's last position: refill it
          named_bar_sync(kKeyDqBar, kKeyDqThreads);
          kfreed = rs + 1;
          if (gi == 0) top_up();
        }
      }
      if (ok) kmore = iter_next<kSub>(kc, a, u1);
    }
    if (gi == 0) {
      volatile uint32_t no_abort = 0;
      for (uint32_t q = kwaited; q < kip; ++q)
        mbar_wait(b_kstage + 8 * (q % NKS), (q / NKS) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    }
  } else if (FP8 && C::kRawRows && warp == 2) {
    // ============================================================ FP8 whole-row key stages
    // Every tile's 128 key rows as two TMA boxes (one per 64-row page half) of all 9 chunks,
    // each half into a stage once the PV MMAs of the tile that used it before have completed
    // over that half's keys. The QK^T MMAs read the stage's keys and the PV MMAs its values
    // (the first 8 chunks of each row). On a tile
    // that ends inside a 32-key MMA step the warp loads the stage on its own barrier and
    // zeroes the rows from the sequence end to the end of that step (the cache may hold NaN
    // there, and 0 * NaN is NaN inside the MMA; those keys are masked) before it signals.
    TileIter it;
    bool more = iter_begin<kSub>(it, a, u0, u1);
    bool ok = true;
    uint32_t p = 0, aux = 0;
    const uint32_t box_bytes = (C::kKStageBytes / 128) * box_rows;
    while (more && ok) {
      const int valid = it.U.L - it.tile * kTileTokens;
      const bool tail = valid < kTileTokens && (valid & 31) != 0;
      const uint32_t sl = p % NKS;
      const uint32_t bar = tail ? b_vaux : b_kstage + 8 * sl, dst = sKS + sl * C::kKStageBytes;
      for (int h = 0; h < 2 && ok; ++h) {
        ok = wait_warp(b_ksfree + 8 * (2 * sl + h), ((p / NKS) & 1) ^ 1);
        if (!ok) break;
        if (lane == 0) {
          if (h == 0) mbar_arrive_expect_tx(bar, it.boxes() * box_bytes);
          load_half<kSub>(it, a, h, &a.tm_k, dst + h * (C::kKStageBytes / 2), bar, 0, box_bytes);
        }
      }
      if (!ok) break;
      if (tail) {
        ok = wait_warp(b_vaux, aux & 1);
        ++aux;
        if (!ok) break;
        // stage [2 halves][8 groups][9 chunks][8 rows][64 B]: the rows' 8 value chunks
        const int nrow = ((valid + 31) & ~31) - valid;
        uint8_t* g = gKS + sl * C::kKStageBytes;
        for (int idx = lane; idx < nrow * 32; idx += 32) {
          const int row = valid + (idx >> 5), c = (idx >> 2) & 7, u16 = idx & 3;
          *reinterpret_cast<uint4*>(g + (row >> 6) * (9 * 4096) + ((row >> 3) & 7) * (9 * 512) + c * 512 +
                                    (row & 7) * 64 + u16 * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_kstage + 8 * sl);
      }
      ++p;
      more = iter_next<kSub>(it, a, u1);
    }
    if (lane == 0) {
      volatile uint32_t no_abort = 0;
      for (uint32_t q = p > (uint32_t)NKS ? p - NKS : 0; q < p; ++q)
        mbar_wait(b_kstage + 8 * (q % NKS), (q / NKS) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    }
  } else if (FP8 && warp == 2) {
    // ============================================================ FP8 raw value producer
    // Every tile's values as two stages of 4 chunks (256 value columns of its 128 rows),
    // each two TMA boxes (one per 64-row page half), which the PV MMAs read as they landed.
    // On a tile that ends inside a 32-key MMA step the warp loads each stage on its own
    // barrier and zeroes the rows from the sequence end to the end of that step (the cache
    // may hold NaN there, and 0 * NaN is NaN inside the MMA) before it signals the stage.
    TileIter it;
    bool more = iter_begin<kSub>(it, a, u0, u1);
    bool ok = true;
    uint32_t p = 0, aux = 0;
    constexpr int kVC = C::kVRawChunks;
    const uint32_t box_bytes = (C::kVStage / 128) * box_rows;
    while (more && ok) {
      const int valid = it.U.L - it.tile * kTileTokens;
      const bool tail = valid < kTileTokens && (valid & 31) != 0;
      for (int j = 0; j < kPairsPerTile; j += C::kPairsPerVStage, ++p) {
        // stage p: value chunks 2j .. 2j + kVC - 1 of the tile's rows
        const uint32_t sl = p % NVS;
        ok = wait_warp(b_vsempty + 8 * sl, ((p / NVS) & 1) ^ 1);
        if (!ok) break;
        const uint32_t bar = tail ? b_vaux : b_vstage + 8 * sl, dst = sVS + sl * C::kVStage;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar, it.boxes() * box_bytes);
          for (int h = 0; h < 2; ++h)
            load_half<kSub>(it, a, h, &a.tm_v, dst + h * (C::kVStage / 2), bar, 2 * j, box_bytes);
        }
        if (tail) {
          ok = wait_warp(b_vaux, aux & 1);
          ++aux;
          if (!ok) break;
          // stage [2 halves][8 groups][kVC chunks][8 rows][64 B]: whole 64-byte rows
          const int nrow = ((valid + 31) & ~31) - valid;
          uint8_t* g = gVS + sl * C::kVStage;
          for (int idx = lane; idx < nrow * kVC * 4; idx += 32) {
            const int row = valid + idx / (kVC * 4), c = (idx >> 2) % kVC, u16 = idx & 3;
            *reinterpret_cast<uint4*>(g + (row >> 6) * (kVC * 4096) + ((row >> 3) & 7) * (kVC * 512) + c * 512 +
                                      (row & 7) * 64 + u16 * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_vstage + 8 * sl);
        }
      }
      if (ok) more = iter_next<kSub>(it, a, u1);
    }
    if (lane == 0) {
      volatile uint32_t no_abort = 0;
      for (uint32_t q = p > (uint32_t)NVS ? p - NVS : 0; q < p; ++q)
        mbar_wait(b_vstage + 8 * (q % NVS), (q / NVS) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    }
  }

  // ============================================================ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

template <int RC, bool FP8, bool kSub>
static cudaError_t prepare_variant() {
  using C = Cfg<RC, FP8>;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<RC, FP8, kSub>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, decode_kernel<RC, FP8, kSub>);
  if (e != cudaSuccess) return e;
  if ((int)attr.sharedSizeBytes > kStaticBudget) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

template <int RC, bool FP8>
static cudaError_t prepare_one() {
  const cudaError_t e = prepare_variant<RC, FP8, false>();
  return e != cudaSuccess ? e : prepare_variant<RC, FP8, true>();
}

template <int RC, bool FP8>
static cudaError_t launch_one(const DecodeArgs& a, int grid, cudaStream_t s) {
  using C = Cfg<RC, FP8>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kDynBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the scheduler
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // pages smaller than 64 rows take the kernel that loads a 64-key block as several boxes
  return a.box_rows < 64 ? cudaLaunchKernelEx(&cfg, decode_kernel<RC, FP8, true>, a)
                         : cudaLaunchKernelEx(&cfg, decode_kernel<RC, FP8, false>, a);
}

int decode_value_chunks_per_box(int rc, bool fp8) {
  switch (rc * 2 + (fp8 ? 1 : 0)) {
    case 33: return Cfg<16, true>::kVRawChunks;
    case 65: return Cfg<32, true>::kVRawChunks;
    case 129: return Cfg<64, true>::kVRawChunks;
    default: return 2;
  }
}

int decode_key_chunks_per_slot(int rc, bool fp8) {
  switch (rc * 2 + (fp8 ? 1 : 0)) {
    case 32: return Cfg<16, false>::KC;
    case 33: return Cfg<16, true>::kKRawChunks;
    case 64: return Cfg<32, false>::KC;
    case 65: return Cfg<32, true>::kKRawChunks;
    case 128: return Cfg<64, false>::KC;
    case 129: return Cfg<64, true>::kKRawChunks;
    default: return 0;
  }
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
