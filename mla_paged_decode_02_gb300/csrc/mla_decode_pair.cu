// mla_decode_pair.cu — paged MLA decode for 128 query rows per key pass, on CTA pairs
// (sm_103a: a cluster of two CTAs on two SMs, tcgen05 MMAs with cta_group::2).
//
// The operation is the one of mla_decode.cu ("[WIP][Attention] FlashAttn MLA", opening
// post: MLA decode as multi-query attention over the shared latent cache; shapes from the
// kernel-test log in "[Attention] Blackwell FP8 MLA support with CUTLASS_MLA backend").
// It serves sequences with more than 64 query rows (s_q * H), above all the 128-head
// DeepSeek-V3 shape that the Blackwell CUTLASS kernel of "[NVIDIA] Add Cutlass MLA
// backend" is built around (its review thread: num_heads must be 128).
//
// Why a pair. For 128 query rows, O^T (512 value columns x 128 rows, float32) fills the
// whole tensor memory of one SM, leaving nothing for the scores; a single CTA must split
// the rows and read every key tile twice. Two SMs together have room for both: a pair
// takes a 256-key super-tile for all 128 rows of a sequence.
//   QK^T (M = 256 keys, N = 128 rows, K = 576): CTA k holds keys 128k..128k+127 of the
//        super-tile as A and query rows 64k..64k+63 as B; its tensor memory receives S^T
//        for its own 128 keys x all 128 rows (128 columns, double-buffered).
//   PV   (M = 256 value columns, N = 128 rows, K = 256 keys), two M-tiles j: CTA k holds
//        value columns 256k+128j..+127 of all 256 keys as A and P^T of rows 64k..64k+63
//        as B; its tensor memory receives O^T for its 256 value columns x 128 rows.
// Tensor memory per CTA: 2 x 128 (S^T) + 2 x 128 (O^T) = 512 columns. Every key byte is
// read from DRAM once per 128 rows; the value columns a CTA needs of its peer's keys come
// from L2 (the peer has just read them).
//
// The FP8 cache. The MMAs read the E4M3 bytes of the cache as TMA lands them (kind::f8f6f4,
// E4M3 x E4M3 with float32 accumulation; the product of two E4M3 values is exact in
// float32), so no thread converts a key or a value. The other operand of an MMA must then be
// E4M3 as well; q and P are each written as two E4M3 terms whose sum keeps the precision
// the result needs:
//   q: this CTA's 64 rows of a unit are scaled per row by a power of two 2^e that puts the
//      row's largest |q| in [128, 256), and q' = q 2^e is stored as hi = e4m3(q') and
//      lo = e4m3(q' - hi). For a bf16 q the sum is exact wherever lo stays a normal E4M3
//      number (|q'| >= 2^-2); smaller entries are off by at most 2^-10 in q' units (2^-17 of
//      the row's largest). S = K.hi + K.lo, and the softmax multiplies row r by 2^-e_r.
//   P: computed times 2^4 (so at most 2^8 with the lazy rescale threshold of 2^4 below) and
//      split the same way from its fp16 rounding: about 8 significant bits, as bf16 P has.
// Each MMA of the bf16 kernel (K = 16) thus becomes two of K = 32: the same tensor time for
// half the bytes.
//
// Softmax coupling. Both CTAs' keys accumulate into the same O^T rows, so they share one
// reference maximum per row. Each CTA runs two softmax warpgroups, warpgroup w for rows
// 64w..64w+63 (one thread per key = one TMEM lane). Per tile the warpgroup tells the
// same warpgroup of the peer whether any of its scores exceeds the reference by more than
// the rescale threshold (and, only then, its row maxima) through distributed shared
// memory; both then move the reference identically. P^T rows 64w.. go to CTA w's P^T
// buffer (its own, or the peer's: bf16 by one bulk copy, FP8 by st.async). At the end of a unit the row sums are
// exchanged the same way; with the FP8 cache the row factors 2^-e too, at its start.
//
// Pipeline per CTA (384 threads). Warp 0: producer, plus each unit's Q. bf16: one ring of
// 32 KB slots in the order the MMAs consume them (the key slots of tile n, then the value
// slots of tile n-1; a unit's last value slots right after its last key slots). FP8: a key
// tile of this CTA's 128 keys as whole 576-byte rows, loaded once the previous tile's QK^T
// is done, and a ring of two 16 KB value blocks one tile behind, fed by one polling thread.
// A TMA load's cost grows with the number of contiguous row pieces in its box (measured on
// this GPU: about 22 GB/s per SM for 128-byte pieces from L2, 44 for 256, 87 for 512), so
// bf16 key boxes take 256-byte pieces of each row (two 64-column chunks), E4M3 key boxes
// whole rows, and value boxes four chunks. Every key and value load completes on the even CTA's barrier, which
// the even CTA alone arms with the bytes of both CTAs (it knows which key halves its peer
// loads), so that no load needs a cross-CTA arrival (each costs a fraction of a
// microsecond). Warp 1 of the even CTA: the single MMA issuer, in program order QK^T(n),
// PV(n-1), QK^T(n+1), ..., a unit's last PV before the next unit's first QK^T (so that the
// epilogue need not wait for it); its commits arrive on the barrier at the same offset in
// both CTAs. Warps 2-3 (FP8): turn each unit's bf16 Q into hi and lo in place. Warps 4-7
// and 8-11: softmax warpgroups 0 and 1, then the epilogue. Every wait is bounded; a stall
// sets the device error word, and both CTAs drain and leave through a final cluster
// barrier.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "mla_internal.h"
#include "mla_pages.cuh"
#include "mla_ptx.cuh"
#include "../../include/mla.h"

namespace mla {
namespace {

constexpr int kPairKeys = 256;              // keys per super-tile
constexpr int kSlotBytes = 32768;           // ring slot
constexpr int kQChunk = 8192;               // 64 rows x 64 columns bf16
constexpr int kPairQBytes = 9 * kQChunk;    // this CTA's 64 query rows: bf16, or E4M3 hi and lo
constexpr int kPairPBytes = kPairKeys * 128;  // P^T for 256 keys x 64 rows: bf16, or E4M3 hi and lo
constexpr int kStageBytes = 16384;         // P^T rows bound for the peer: 128 keys x 64 rows
constexpr int kRing = 3;                    // bf16: ring of key and value slots
constexpr int kVRing = 2;                   // FP8: ring of 16 KB value blocks
constexpr int kKTileBytes = 2 * 36864;      // FP8: this CTA's 128 keys as whole 576-byte rows
constexpr int kVBlockBytes = 16384;         // FP8: 64 keys x this CTA's 256 value columns
constexpr int kPairThreads = 384;
constexpr int kPairTmemCols = 512;
constexpr int kOCol = 256;                  // O^T M-tile j at columns 256 + 128 j
constexpr float kPLog2e = 1.4426950408889634f;
constexpr float kPLn2 = 0.6931471805599453f;
constexpr int kPairSmemLimit = 232448;
constexpr int kPairStaticBudget = 9216;
// bf16: Q, P^T, the staging buffer of P^T rows bound for the peer, the ring. FP8: Q, P^T, the
// key tile, the value ring (P^T rows for the peer go by st.async).
constexpr int kPairDynBytes16 = 1024 + kPairQBytes + kPairPBytes + kStageBytes + kRing * kSlotBytes;
constexpr int kPairDynBytes8 = 1024 + kPairQBytes + kPairPBytes + kKTileBytes + kVRing * kVBlockBytes;
constexpr int pair_dyn_bytes(bool fp8) { return fp8 ? kPairDynBytes8 : kPairDynBytes16; }
static_assert(kPairDynBytes16 + kPairStaticBudget <= kPairSmemLimit, "shared memory budget");
static_assert(kPairDynBytes8 + kPairStaticBudget <= kPairSmemLimit, "shared memory budget");

// The bf16 ring's slot plan: a key slot is KC = 2 adjacent 64-column chunks of this CTA's
// 128 keys ([2 halves][8 groups][2 chunks][8 rows][128 B], 5 slots per super-tile, the last
// holding chunk 8 and a zero-filled chunk past the row, which TMA fills); a value slot is
// this CTA's 256 value columns of one 64-key block ([8 groups][4 chunks][8 rows][128 B]).
// E4M3 value blocks have the same shape with 64-byte row pieces. Per cache type also the
// softmax's lazy rescale threshold and the power of two P is computed times.
template <bool FP8>
struct PairCfg {
  static constexpr int kKeyChunks = 2;
  static constexpr int kKeySlots = 5;
  static constexpr int kRowBytes = FP8 ? 64 : 128;      // one chunk of one row
  static constexpr int kBlockBytes = kSlotBytes;        // bf16: one 64-key value block per slot
  static constexpr float kRescaleLog2 = FP8 ? 4.f : 8.f;  // lazy rescale threshold (log2 units)
  static constexpr float kPOffLog2 = FP8 ? 4.f : 0.f;     // P is computed times 2^kPOffLog2
  static_assert(FP8 || 4 * 8 * kRowBytes * 8 == kBlockBytes, "value block layout");
  static_assert(FP8 || kKeyChunks * 8 * kRowBytes == 2048, "key slot group stride");
  static_assert(kKeySlots * kKeyChunks >= 9, "a tile is 9 chunks");
};

struct PUnit {
  int b, g, tb, te, slot, L;
};

__device__ __forceinline__ PUnit load_punit(const DecodeArgs& a, int u) {
  const int4 v = a.units[u];
  PUnit r;
  r.b = v.x;
  r.g = v.y;
  r.tb = v.z & 0xFFFF;
  r.te = (int)((unsigned)v.z >> 16);
  r.slot = v.w;
  r.L = a.batch_info[r.b].z;
  return r;
}

// First global cache row of each 64-key block kb of super-tile `tile` (-1: past the
// sequence end). A block-table entry outside the pool is flagged and reads page 0.
// kSub: pages smaller than 64 rows (boxes of a.box_rows rows), else one box per block.
template <bool kSub>
__device__ __forceinline__ void block_rows(const DecodeArgs& a, const PUnit& U, int tile, int64_t* rb, int* nb) {
  const int32_t* bt = a.block_table + (int64_t)U.b * a.MB;
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    const int tok = tile * kPairKeys + 64 * kb;
    rb[kb] = tok < U.L ? page_row(bt, tok, a) : -1;
    nb[kb] = kSub ? block_boxes(U.L - tok, a.box_rows) : (tok < U.L ? 1 : 0);
  }
}

// The page numbers of the four 64-key blocks of super-tile `tile` (the block-table index
// clamped to the row, so that the load is safe past the sequence end), loaded ahead of use.
__device__ __forceinline__ void tile_pages(const DecodeArgs& a, int b, int tile, int* pg) {
  const int32_t* bt = a.block_table + (int64_t)b * a.MB;
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) pg[kb] = __ldg(bt + min((tile * kPairKeys + 64 * kb) / a.P, a.MB - 1));
}

// block_rows from page numbers loaded before: the same rows and box counts.
template <bool kSub>
__device__ __forceinline__ void rows_from_pages(const DecodeArgs& a, int L, int tile, const int* pg, int64_t* rb,
                                                int* nb) {
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    const int tok = tile * kPairKeys + 64 * kb;
    const int off = tok % a.P;
    rb[kb] = tok >= L ? -1 : (pg[kb] < 0 || pg[kb] >= a.num_pages) ? (int64_t)off : (int64_t)pg[kb] * a.P + off;
    nb[kb] = kSub ? block_boxes(L - tok, a.box_rows) : (tok < L ? 1 : 0);
  }
}

// The rows of a key tile, kept for the value loads of the same tile that follow it.
struct TileRows {
  int64_t rb[4];
  int nb[4];
  int L, b, tile;
};
constexpr int kRowsQ = 4;   // key tiles whose values are not all loaded: at most 3

__device__ __forceinline__ uint32_t p_off128(int row, int u) {   // 128-byte swizzled bf16 P^T row
  return (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u + ((uint32_t)(u ^ (row & 7)) << 4);
}
__device__ __forceinline__ uint32_t p_off64(int row, int u) {    // 64-byte swizzled E4M3 P^T row
  return (uint32_t)(row >> 3) * 512u + (uint32_t)(row & 7) * 64u + ((uint32_t)(u ^ ((row >> 1) & 3)) << 4);
}

// 4 x 4 transpose inside each quad of lanes: lane j of the quad holds a[i] = M[i][j] before
// and a[k] = M[j][k] after (2 x 2 blocks first, then the blocks).
__device__ __forceinline__ void quad_transpose4(uint32_t* a, int j) {
  const bool odd = (j & 1) != 0, up = (j & 2) != 0;
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    const uint32_t r = __shfl_xor_sync(0xffffffffu, odd ? a[i] : a[i + 1], 1);
    if (odd) a[i] = r;
    else a[i + 1] = r;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t r = __shfl_xor_sync(0xffffffffu, up ? a[i] : a[i + 2], 2);
    if (up) a[i] = r;
    else a[i + 2] = r;
  }
}

// Non-blocking test of an mbarrier phase (a producer polling two rings).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace

template <bool FP8, bool kSub>
__global__ void __launch_bounds__(kPairThreads, 1) decode_pair_kernel(const __grid_constant__ DecodeArgs a) {
  using Cfg = PairCfg<FP8>;
  constexpr int KC = Cfg::kKeyChunks, kKeySlots = Cfg::kKeySlots;
  extern __shared__ uint8_t dsmem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kRing], bar_empty[kRing], bar_aux;
  __shared__ __align__(8) uint64_t bar_qfull, bar_qempty;
  // FP8: Q landed (this CTA), Q converted (both CTAs, on the even CTA), this CTA's row
  // factors written and read
  __shared__ __align__(8) uint64_t bar_qraw, bar_qready, bar_qsc, bar_qfree;
  __shared__ __align__(8) uint64_t bar_ktfull, bar_ktempty;   // FP8: the key tile
  __shared__ __align__(16) uint32_t sig_s[4];        // landing place of the odd CTA's 16-byte signals
  __shared__ __align__(8) uint64_t bar_sfull[2], bar_sempty[2], bar_pfull, bar_pin, bar_pvdone, bar_oempty;
  __shared__ __align__(8) uint64_t bar_x[2][2];
  __shared__ __align__(8) uint64_t bar_drain, bar_never;
  __shared__ uint32_t tmem_base_s, abort_s;
  __shared__ __align__(16) float xbuf[2][2][68];     // [warpgroup][parity]: word 0 flag, words 4..67 values
  __shared__ __align__(16) float mref_s[2][64];
  __shared__ __align__(16) float rowc_s[2][64];     // FP8: score factor of each row (log2 units)
  __shared__ float qf_s[64];                        // FP8: 2^-e of this CTA's 64 query rows
  __shared__ float alpha_s[2][64], own_s[2][64];
  __shared__ int nvis_s[2][64];
  __shared__ TileRows rows_q[kRowsQ];               // FP8 producer: rows of issued key tiles
  __shared__ float wred_s[2][4][64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;

  const uint32_t raw = smem_u32(dsmem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = dsmem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sP = sQ + kPairQBytes;
  const uint32_t sStage = sP + kPairPBytes;                     // bf16
  const uint32_t sKT = sP + kPairPBytes;                        // FP8: key tile
  const uint32_t sR = FP8 ? sKT + kKTileBytes : sStage + kStageBytes;   // the (value) ring
  uint8_t* gQ = gbase;
  uint8_t* gP = gbase + kPairQBytes;
  uint8_t* gStage = gP + kPairPBytes;
  uint8_t* gR = gbase + (sR - sQ);

  const uint32_t b_full = smem_u32(bar_full), b_empty = smem_u32(bar_empty), b_aux = smem_u32(&bar_aux);
  const uint32_t b_qfull = smem_u32(&bar_qfull), b_qempty = smem_u32(&bar_qempty);
  const uint32_t b_qraw = smem_u32(&bar_qraw), b_qready = smem_u32(&bar_qready);
  const uint32_t b_qsc = smem_u32(&bar_qsc), b_qfree = smem_u32(&bar_qfree);
  const uint32_t b_ktfull = smem_u32(&bar_ktfull), b_ktempty = smem_u32(&bar_ktempty);
  const uint32_t b_sfull = smem_u32(bar_sfull), b_sempty = smem_u32(bar_sempty);
  const uint32_t b_pfull = smem_u32(&bar_pfull), b_pin = smem_u32(&bar_pin), b_pvdone = smem_u32(&bar_pvdone);
  const uint32_t b_oempty = smem_u32(&bar_oempty), b_drain = smem_u32(&bar_drain);
  const uint32_t b_x = smem_u32(bar_x);
  const uint32_t b_never = smem_u32(&bar_never);   // tests: a barrier nothing arrives on
  volatile uint32_t* abort_flag = &abort_s;
  uint32_t* err = a.err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(b_full + 8 * i, 1);       // the even CTA's producer, with both CTAs' bytes
      mbar_init(b_empty + 8 * i, 1);
    }
    mbar_init(b_aux, 1);
    mbar_init(b_qfull, 1);                // bf16: the even CTA's arrival, with both CTAs' bytes
    mbar_init(b_qempty, 1);
    mbar_init(b_qraw, 1);                 // FP8: this CTA's producer, with its bytes
    mbar_init(b_qready, 1);               // FP8: the even CTA's converters, expecting the odd CTA's 16-byte signal
    mbar_init(b_qsc, 1);                  // FP8: this CTA's converters
    mbar_init(b_qfree, 1);                // FP8: the softmax warpgroup of this CTA's rows
    mbar_init(b_ktfull, 1);               // FP8: the even CTA's producer, with both CTAs' bytes
    mbar_init(b_ktempty, 1);              // FP8: the MMA issuer's commit (both CTAs)
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_sempty + 8 * i, 2);     // the even CTA's two warpgroups (the odd CTA's
    }                                     // reads precede its P^T signals)
    // P^T of a tile is complete in both CTAs: the even CTA's warpgroup 0 (its own rows, and
    // it expects the odd CTA's bulk copy of rows for the even CTA's P^T) and the odd CTA's
    // warpgroup 1 (its own rows, once the even CTA's copy into its P^T has landed on b_pin)
    mbar_init(b_pfull, 2);
    mbar_init(b_pin, 1);
    mbar_init(b_pvdone, 1);
    mbar_init(b_oempty, 2);               // the even CTA's two warpgroups, as b_sempty
    for (int i = 0; i < 4; ++i) mbar_init(b_x + 8 * i, 1);   // own arrival + the peer's bytes
    mbar_init(b_drain, 1);
    mbar_init(b_never, 1);
    abort_s = 0u;
    fence_mbarrier_init();
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
  }
  if (warp == 0) tmem_alloc_pair(smem_u32(&tmem_base_s), kPairTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();                         // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  griddep_wait();

  const int u0 = a.cta_first[pair], u1 = a.cta_first[pair + 1];
  const int R = a.R;
  auto lead = [&](uint32_t addr) { return map_to_rank(addr, 0); };
  // A failed wait also raises the peer's abort flag, so that its waits end too.
  auto fail_peer = [&]() { st_cluster_u32(map_to_rank(smem_u32(&abort_s), peer), 1u); };
  auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = mbar_wait(bar, parity, abort_flag, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    if (!ok) fail_peer();
    return ok;
  };

  if (warp < 4) {
    if (warp == 0) {
      if constexpr (FP8) {
      // ================================================================ producer (FP8)
      // One thread feeds three streams, polling their barriers: each unit's Q (this CTA's 64
      // rows, on this CTA's barrier for its converters); the key tiles — this CTA's 128 keys
      // of a super-tile as whole 576-byte rows, one TMA row piece per key, into the single key
      // tile once the previous tile's QK^T MMAs are done with it; and the value blocks (64 keys
      // x this CTA's 256 value columns) into a ring of two, one key tile behind, so that they
      // read rows the key loads have brought into L2.
      if (lane == 0) {
        const uint64_t pol_keep = l2_policy_evict_last(), pol_last = l2_policy_evict_first();
        const uint32_t box_rows = kSub ? (uint32_t)a.box_rows : 64u;
        const uint32_t kbox_bytes = kDQK * box_rows;           // one whole-row key box
        const uint32_t vbox_bytes = 256 * box_rows;             // one 4-chunk value box
        uint32_t nq = 0, nkt = 0, rv = 0, aux = 0, vseq = 0;
        int ku = u0, kt = 0, vkb = 0;
        bool kq = true, kdone = u0 >= u1;
        // Loads are issued well before their values are used, so that the one thread feeding
        // three streams does not wait on them: the next unit's descriptor (its length one unit
        // ahead, the raw descriptor two ahead) and the page numbers of the next key tile.
        PUnit KU{}, KN{};
        int4 n4 = make_int4(0, 0, 0, 0);
        int kpg[4] = {0, 0, 0, 0};
        auto next_unit = [&](int u) {           // KN <- unit u + 1 (from n4), n4 <- unit u + 2
          KN.b = n4.x;
          KN.g = n4.y;
          KN.tb = n4.z & 0xFFFF;
          KN.te = (int)((unsigned)n4.z >> 16);
          KN.slot = n4.w;
          KN.L = u + 1 < u1 ? __ldg(&a.batch_info[n4.x].z) : 0;
          n4 = u + 2 < u1 ? __ldg(&a.units[u + 2]) : make_int4(0, 0, 0, 0);
        };
        if (!kdone) {
          KU = load_punit(a, u0);
          if (u0 + 1 < u1) n4 = __ldg(&a.units[u0 + 1]);
          next_unit(u0);
          kt = KU.tb;
          tile_pages(a, KU.b, kt, kpg);
        }
        uint64_t t_last = global_timer_ns();
        while (!(kdone && vseq == nkt)) {
          bool prog = false;
          if (!kdone) {
            if (kq) {
              if (mbar_test(b_qempty, (nq & 1) ^ 1)) {
                const int32_t qg = (128 * KU.g + 64 * (int)rank) / 8, q0 = 128 * KU.g + 64 * (int)rank;
                mbar_arrive_expect_tx(b_qraw, kPairQBytes);
                if (a.q_whole_rows)     // one box of 64 whole rows: [8 groups][9 chunks][8 rows][128 B]
                  tma_load_5d_hint(sQ, &a.tm_q, b_qraw, 0, 0, 0, qg, KU.b, pol_keep);
                else                    // 9 boxes of one 64-column chunk: [9 chunks][64 rows][128 B]
                  for (int c = 0; c < 9; ++c) tma_load_3d_hint(sQ + c * kQChunk, &a.tm_q, b_qraw, 64 * c, q0, KU.b, pol_keep);
                ++nq;
                kq = false;
                prog = true;
              }
            } else if (mbar_test(b_ktempty, (nkt & 1) ^ 1)) {
              TileRows& e = rows_q[nkt % kRowsQ];
              int64_t rb[4];
              int nb[4];
              rows_from_pages<kSub>(a, KU.L, kt, kpg, rb, nb);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                e.rb[i] = rb[i];
                e.nb[i] = nb[i];
              }
              e.L = KU.L;
              e.b = KU.b;
              e.tile = kt;
              const int32_t* bt = a.block_table + (int64_t)KU.b * a.MB;
              // every key tile takes bytes from both CTAs (see the bf16 ring below)
              const int nown = nb[2 * rank] + nb[2 * rank + 1], nodd = nb[2] + nb[3];
              const uint32_t nbox = (uint32_t)(nb[0] + nb[1] + (nodd > 0 ? nodd : 1));
              const uint32_t lb = lead(b_ktfull);
              if (leader) mbar_arrive_expect_tx(b_ktfull, nbox * kbox_bytes);
              if (nown == 0) tma_load_4d_pair_hint(sKT, &a.tm_k, lb, 0, 0, 0, (int32_t)(rb[0] >> 3), pol_keep);
              for (int h = 0; h < 2; ++h) {
                const int kb = 2 * (int)rank + h;
                if (nb[kb] == 0) continue;
                const uint32_t d = sKT + h * (kKTileBytes / 2);
                tma_load_4d_pair_hint(d, &a.tm_k, lb, 0, 0, 0, (int32_t)(rb[kb] >> 3), pol_keep);
                if (kSub && nb[kb] > 1)
                  load_more_boxes(kBoxPairHint, &a.tm_k, d, lb, 0, kbox_bytes, bt, a, kt * kPairKeys + 64 * kb, nb[kb],
                                  pol_keep);
              }
              ++nkt;
              prog = true;
              if (++kt == KU.te) {
                if (++ku == u1) {
                  kdone = true;
                } else {
                  KU = KN;
                  next_unit(ku);
                  kt = KU.tb;
                  kq = true;
                }
              }
              if (!kdone) tile_pages(a, KU.b, kt, kpg);
            }
          }
          // value block vkb of key tile vseq, once the next key tile has been issued (so this
          // tile's key rows have landed) or the keys are done
          if (vseq + 1 < nkt || (kdone && vseq < nkt)) {
            const uint32_t slot = rv % kVRing;
            if (mbar_test(b_empty + 8 * slot, ((rv / kVRing) & 1) ^ 1)) {
              const TileRows& e = rows_q[vseq % kRowsQ];
              const int kb = vkb;
              const int valid = e.L - e.tile * kPairKeys - 64 * kb;
              const int tok0 = e.tile * kPairKeys + 64 * kb;
              const int32_t* vbt = a.block_table + (int64_t)e.b * a.MB;
              const int64_t vrb = e.rb[kb];
              const int vnb = e.nb[kb];
              // a block not loaded whole (32-key MMA steps past the end, or boxes past it) is
              // loaded here first, its rows up to the end of the last step zeroed (the cache may
              // hold NaN there, and 0 * NaN is NaN inside the MMA), then its bytes counted
              const bool zero = valid < 64 && ((valid & 31) != 0 || (kSub && vnb < (int)(64 / box_rows)));
              const uint32_t lb = lead(b_full + 8 * slot), dst = sR + slot * kVBlockBytes;
              const int32_t c0 = 4 * (int)rank;               // this CTA's value columns 256 rank ..
              if (leader) mbar_arrive_expect_tx(b_full + 8 * slot, 2u * kVBlockBytes);
              bool vok = true;
              if (!zero) {
                tma_load_4d_pair_hint(dst, &a.tm_v, lb, 0, 0, c0, (int32_t)(vrb >> 3), pol_last);
                if (kSub && vnb > 1)
                  load_more_boxes(kBoxPairHint, &a.tm_v, dst, lb, c0, vbox_bytes, vbt, a, tok0, vnb, pol_last);
              } else {
                mbar_arrive_expect_tx(b_aux, (kSub ? (uint32_t)vnb : 1u) * vbox_bytes);
                tma_load_4d_hint(dst, &a.tm_v, b_aux, 0, 0, c0, (int32_t)(vrb >> 3), pol_last);
                if (kSub && vnb > 1)
                  load_more_boxes(kBoxHint, &a.tm_v, dst, b_aux, c0, vbox_bytes, vbt, a, tok0, vnb, pol_last);
                vok = wait(b_aux, aux & 1);
                ++aux;
                if (vok) {
                  // block [8 key groups][4 chunks][8 rows][64 B]: zero whole rows
                  const int nrow = ((valid + 31) & ~31) - valid;
                  uint8_t* g = gR + slot * kVBlockBytes;
                  for (int idx = 0; idx < nrow * 16; ++idx) {
                    const int row = valid + (idx >> 4), c = (idx >> 2) & 3, u16 = idx & 3;
                    *reinterpret_cast<uint4*>(g + (row >> 3) * 2048 + c * 512 + (row & 7) * 64 + u16 * 16) =
                        make_uint4(0, 0, 0, 0);
                  }
                  fence_proxy_async_smem();
                  fence_acq_rel_cluster();
                  mbar_complete_tx_cluster(lb, kVBlockBytes);   // this CTA's share of the block is in place
                }
              }
              if (!vok) break;
              ++rv;
              prog = true;
              if (++vkb == 4 || valid <= 64) {
                vkb = 0;
                ++vseq;
              }
            }
          }
          if (prog) {
            t_last = global_timer_ns();
          } else {
            if (*abort_flag) break;
            if (global_timer_ns() - t_last > a.wait_limit_ns) {
              *abort_flag = 1u;
              atomicOr(err, MLA_DEVERR_TIMEOUT);
              fail_peer();
              break;
            }
          }
        }
        if (*abort_flag) {     // see below: the odd CTA cannot observe its own loads then
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 50000ull) {
          }
        }
        // no copy into this CTA's memory may be in flight when it leaves
        volatile uint32_t no_abort = 0;
        if (leader) {
          if (nkt > 0)
            mbar_wait(b_ktfull, (nkt - 1) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
          for (uint32_t q = rv > (uint32_t)kVRing ? rv - kVRing : 0; q < rv; ++q)
            mbar_wait(b_full + 8 * (q % kVRing), (q / kVRing) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
        }
        if (nq > 0) mbar_wait(b_qraw, (nq - 1) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
      }
      } else {
      // ================================================================ producer
      // Ring order per super-tile n: its key slots (chunks KC ks .. KC ks + KC - 1 of this
      // CTA's 128 keys each), then the value slots of tile n-1 (this CTA's 256 value columns
      // of the 64-key blocks before the sequence end); a unit's last value slots follow its
      // last key slots.
      uint32_t r = 0, uq = 0, aux = 0;
      bool ok = true;
      // a key's lines are read again (as values, by this CTA or its peer) about one tile later:
      // keep them in L2; the value read is their last use
      const uint64_t pol_keep = l2_policy_evict_last(), pol_last = l2_policy_evict_first();
      const int32_t* bt_all = a.block_table;
      const uint32_t box_rows = kSub ? (uint32_t)a.box_rows : 64u;             // rows of one box
      const uint32_t kbox_bytes = (kSlotBytes / 128) * box_rows;               // one key box
      const uint32_t vbox_bytes = (Cfg::kBlockBytes / 64) * box_rows;          // one value box
      auto load_values = [&](const PUnit& U, int tile, const int64_t* rb, const int* nb) -> bool {
        const int32_t* bt = bt_all + (int64_t)U.b * a.MB;
        for (int kb = 0; kb < 4; ++kb) {
          if (rb[kb] < 0) break;                       // blocks past the sequence end
          const uint32_t slot = r % kRing;
          bool w_ok = lane != 0 || wait(b_empty + 8 * slot, ((r / kRing) & 1) ^ 1);
          if (!__all_sync(0xffffffffu, w_ok)) return false;
          const uint32_t lb = lead(b_full + 8 * slot);
          const int32_t c0 = 4 * (int)rank;            // this CTA's value columns 256 rank ..
          if (leader && lane == 0) mbar_arrive_expect_tx(b_full + 8 * slot, 2u * Cfg::kBlockBytes);
          const int valid = U.L - tile * kPairKeys - 64 * kb;
          // the block holding the sequence end gets its rows up to the end of its last MMA K
          // step zeroed (the cache may hold NaN there, and 0 * NaN is NaN inside the MMA); a
          // block not loaded whole completes its bytes itself
          const bool zero = valid < 64 && ((valid % 16) != 0 || (kSub && nb[kb] < (int)(64 / box_rows)));
          const int tok0 = tile * kPairKeys + 64 * kb;
          const uint32_t dst = sR + slot * kSlotBytes;
          if (!zero) {
            if (lane == 0) {
              tma_load_4d_pair_hint(dst, &a.tm_v, lb, 0, 0, c0, (int32_t)(rb[kb] >> 3), pol_last);
              if (kSub && nb[kb] > 1)
                load_more_boxes(kBoxPairHint, &a.tm_v, dst, lb, c0, vbox_bytes, bt, a, tok0, nb[kb], pol_last);
            }
          } else {
            if (lane == 0) {
              mbar_arrive_expect_tx(b_aux, (kSub ? (uint32_t)nb[kb] : 1u) * vbox_bytes);
              tma_load_4d_hint(dst, &a.tm_v, b_aux, 0, 0, c0, (int32_t)(rb[kb] >> 3), pol_last);
              if (kSub && nb[kb] > 1)
                load_more_boxes(kBoxHint, &a.tm_v, dst, b_aux, c0, vbox_bytes, bt, a, tok0, nb[kb], pol_last);
            }
            w_ok = wait(b_aux, aux & 1);
            ++aux;
            if (!__all_sync(0xffffffffu, w_ok)) return false;
            // block layout [8 key groups][4 chunks][8 rows][128 B]: zero whole rows
            const int nrow = ((valid + 15) & ~15) - valid;   // to the end of the 16-key step
            uint8_t* g = gR + slot * kSlotBytes;
            for (int idx = lane; idx < nrow * 32; idx += 32) {
              const int row = valid + (idx >> 5), c = (idx >> 3) & 3, u16 = idx & 7;
              *reinterpret_cast<uint4*>(g + (row >> 3) * 4096 + c * 1024 + (row & 7) * 128 + u16 * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              fence_acq_rel_cluster();
              mbar_complete_tx_cluster(lb, Cfg::kBlockBytes);   // this CTA's share of the block is in place
            }
          }
          ++r;
        }
        return true;
      };

      PUnit pu{};
      int ptile = -1;
      int64_t prb[4] = {-1, -1, -1, -1};
      int pnb[4] = {0, 0, 0, 0};
      for (int u = u0; u < u1 && ok; ++u, ++uq) {
        const PUnit U = load_punit(a, u);
        // this CTA's 64 query rows of the unit (rows past R read as zeros), kept in L2 for the
        // re-reads of long sequences' units, counted on the even CTA's barrier with both CTAs'
        // bytes: as one box of 64 whole rows ([8 groups][9 chunks][8 rows][128 B]) or as 9
        // boxes of one 64-column chunk ([9 chunks][64 rows][128 B])
        bool w_ok = lane != 0 || wait(b_qempty, (uq & 1) ^ 1);
        ok = __all_sync(0xffffffffu, w_ok);
        if (!ok) break;
        if (lane == 0) {
          const int32_t qg = (128 * U.g + 64 * (int)rank) / 8, q0 = 128 * U.g + 64 * (int)rank;
          const uint32_t lb = lead(b_qfull);
          if (leader) mbar_arrive_expect_tx(b_qfull, 2 * kPairQBytes);
          if (a.q_whole_rows)
            tma_load_5d_pair_hint(sQ, &a.tm_q, lb, 0, 0, 0, qg, U.b, pol_keep);
          else
            for (int c = 0; c < 9; ++c)
              tma_load_3d_pair_hint(sQ + c * kQChunk, &a.tm_q, lb, 64 * c, q0, U.b, pol_keep);
        }
        for (int tile = U.tb; tile < U.te && ok; ++tile) {
          int64_t rb[4];
          int nb[4];
          block_rows<kSub>(a, U, tile, rb, nb);
          const int32_t* bt = bt_all + (int64_t)U.b * a.MB;
          // Bytes of both CTAs' key halves (the even CTA arms the barrier for both). Every key
          // slot needs bytes from both CTAs: the odd CTA's half of a super-tile that lies past
          // the sequence end gets one box of rows the even CTA reads anyway (the softmax masks
          // those keys). Were it to load nothing, the slot could complete on the even CTA's
          // bytes alone and be consumed and released again before the odd producer waits for
          // its previous release, and a parity wait cannot tell those two phases apart.
          const int nown = nb[2 * rank] + nb[2 * rank + 1];   // this CTA's key boxes
          const int nodd = nb[2] + nb[3];
          const uint32_t nbox = (uint32_t)(nb[0] + nb[1] + (nodd > 0 ? nodd : 1));
          for (int ks = 0; ks < kKeySlots; ++ks) {
            const uint32_t slot = r % kRing;
            w_ok = lane != 0 || wait(b_empty + 8 * slot, ((r / kRing) & 1) ^ 1);
            ok = __all_sync(0xffffffffu, w_ok);
            if (!ok) break;
            if (lane == 0) {
              const uint32_t lb = lead(b_full + 8 * slot), dst = sR + slot * kSlotBytes;
              if (leader) mbar_arrive_expect_tx(b_full + 8 * slot, nbox * kbox_bytes);
              if (nown == 0)        // odd CTA, half past the end: one box of the even CTA's first rows
                tma_load_4d_pair_hint(dst, &a.tm_k, lb, 0, 0, KC * ks, (int32_t)(rb[0] >> 3), pol_keep);
              for (int h = 0; h < 2; ++h) {
                const int kb = 2 * (int)rank + h;
                if (nb[kb] == 0) continue;
                const uint32_t d = dst + h * (kSlotBytes / 2);
                tma_load_4d_pair_hint(d, &a.tm_k, lb, 0, 0, KC * ks, (int32_t)(rb[kb] >> 3), pol_keep);
                if (kSub && nb[kb] > 1)
                  load_more_boxes(kBoxPairHint, &a.tm_k, d, lb, KC * ks, kbox_bytes, bt, a, tile * kPairKeys + 64 * kb,
                                  nb[kb], pol_keep);
              }
            }
            ++r;
          }
          if (!ok) break;
          if (ptile >= 0) ok = load_values(pu, ptile, prb, pnb);
          pu = U;
          ptile = tile;
          for (int kb = 0; kb < 4; ++kb) { prb[kb] = rb[kb]; pnb[kb] = nb[kb]; }
        }
        // the unit's last value slots before the next unit's Q and keys (the MMA issuer takes
        // the unit's last PV before the next unit's first QK^T)
        if (ok && ptile >= 0) ok = load_values(pu, ptile, prb, pnb);
        ptile = -1;
      }
      // after an abort the odd CTA cannot observe its own key and value loads (they count on
      // the even CTA's barrier, whose phase may never complete): both producers wait 50 us,
      // far longer than a load takes, before leaving
      if (*abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 50000ull) {
        }
      }
      // a CTA must not leave with copies into its memory in flight: the even CTA waits until
      // the last loads of both CTAs have landed (normally the MMA issuer already has)
      if (lane == 0 && leader) {
        volatile uint32_t no_abort = 0;
        for (uint32_t q = r > (uint32_t)kRing ? r - kRing : 0; q < r; ++q)
          mbar_wait(b_full + 8 * (q % kRing), (q / kRing) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
        if (uq > 0) mbar_wait(b_qfull, (uq - 1) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
      }
      }
    } else if (warp == 1 && leader) {
      // ================================================================ MMA issuer (even CTA)
      if (lane == 0) {
        // The MMA loops are fully unrolled (a partial block leaves early): this one thread
        // issues every MMA of the pair, and its own instructions per MMA set their pace. The
        // loops around them, which wait on barriers, stay rolled (their code would crowd the
        // instruction cache the CTA's roles share).
        // operands bf16 (kind::f16), or E4M3 (kind::f8f6f4: format code 0 is E4M3 there)
        const uint32_t idesc_qk = make_idesc(256, 128, FP8 ? 0u : 1u, 0, 0);
        const uint32_t idesc_pv = make_idesc(256, 128, FP8 ? 0u : 1u, 1, 1);
        constexpr uint32_t kSw = FP8 ? kSwizzle64 : kSwizzle128;
        // key slot [2 halves][8 groups][KC chunks][8 rows][row piece]: K-major, 8-row groups 2 KB apart
        const uint64_t dK0 = make_sdesc(sR, 16, 2048, kSw);
        // Q chunk c: [64 rows][128 B] at sQ + 8 KB c, or chunk c of [8 groups][9 chunks][8 rows][128 B];
        // E4M3: the first (hi) and second (lo) 512 bytes of each of those 1 KB blocks, 64-byte rows
        const uint64_t dQ0 = make_sdesc(sQ, 16, a.q_whole_rows ? 9 * 1024 : 1024, kSw);
        const uint32_t q_chunk = a.q_whole_rows ? 1024 : kQChunk;
        // value block [8 groups][4 chunks][8 rows][row piece]: MN-major, chunks 8 rows apart
        const uint64_t dV0 = make_sdesc(sR, 8 * Cfg::kRowBytes, 32 * Cfg::kRowBytes, kSw);
        // MN-major P^T: bf16 [256 keys][128 B]; E4M3 [key half][hi, lo][128 keys][64 B]
        const uint64_t dP0 = FP8 ? make_sdesc(sP, 512, 512, kSwizzle64) : make_sdesc(sP, 1024, 1024, kSwizzle128);
        // FP8 key tile [16 groups][9 chunks][8 rows][64 B]: K-major, 8-row groups 4.5 KB apart
        const uint64_t dKT0 = make_sdesc(sKT, 16, 9 * 512, kSwizzle64);
        uint32_t r = 0, n = 0, uc = 0, pvn = 0, nkt = 0;
        bool ok = true;
        struct Prev {
          int L, tile;
          bool first;
          uint32_t uc;
        } prev{0, -1, false, 0};
        auto issue_pv = [&](const Prev& pv) -> bool {
          if (!wait(b_pfull, pvn & 1)) return false;
          if (FP8) fence_proxy_async_smem();   // P^T rows that came from the peer by st.async
          if (pv.first && !wait(b_oempty, (pv.uc & 1) ^ 1)) return false;
          if constexpr (FP8) {
            // value blocks of 64 keys from the ring of two
            for (int kb = 0; kb < 4; ++kb) {
              const int valid = pv.L - pv.tile * kPairKeys - 64 * kb;
              if (valid <= 0) break;
              const int ksteps = valid >= 64 ? 2 : (valid + 31) / 32;
              const uint32_t slot = r % kVRing;
              if (!wait(b_full + 8 * slot, (r / kVRing) & 1)) return false;
              tc_fence_after();
              const uint64_t ad = dV0 + (uint64_t)((slot * kVBlockBytes) >> 4);
              // P^T of block kb: key half kb / 2, keys 64 (kb % 2) .. of it; lo 8 KB after hi
              const uint64_t bd = dP0 + (uint64_t)(((kb >> 1) * 16384 + (kb & 1) * 4096) >> 4);
              // M-tile j: this CTA's value columns 128 j .. (its chunks 2j, 2j + 1)
#pragma unroll
              for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                  if (kk >= ksteps) break;
                  const uint64_t aj = ad + (uint64_t)((1024 * j + 8192 * kk) >> 4);
                  const uint64_t bk = bd + (uint64_t)((2048 * kk) >> 4);
                  umma_pair_f8(tmem + kOCol + 128 * j, aj, bk, idesc_pv, !(pv.first && kb == 0 && kk == 0));
                  umma_pair_f8(tmem + kOCol + 128 * j, aj, bk + (8192 >> 4), idesc_pv, 1u);
                }
              umma_pair_commit(b_empty + 8 * slot);
              ++r;
            }
            umma_pair_commit(b_pvdone);
            ++pvn;
            return true;
          } else {
          // bf16: a value slot per 64-key block before the sequence end
          for (int kb = 0; kb < 4; ++kb) {
            const int valid = pv.L - pv.tile * kPairKeys - 64 * kb;
            if (valid <= 0) break;
            const int ksteps = valid >= 64 ? 4 : (valid + 15) / 16;
            const uint32_t slot = r % kRing;
            if (!wait(b_full + 8 * slot, (r / kRing) & 1)) return false;
            tc_fence_after();
            const uint64_t ad = dV0 + (uint64_t)((slot * kSlotBytes) >> 4);
            const uint64_t bd = dP0 + (uint64_t)((64 * kb * 128) >> 4);
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                if (kk >= ksteps) break;
                umma_pair_f16(tmem + kOCol + 128 * j, ad + (uint64_t)((2048 * j + 8192 * kk) >> 4), bd + kk * (2048 >> 4),
                              idesc_pv, !(pv.first && kb == 0 && kk == 0));
              }
            umma_pair_commit(b_empty + 8 * slot);
            ++r;
          }
          umma_pair_commit(b_pvdone);
          ++pvn;
          return true;
          }
        };
        for (int u = u0; u < u1 && ok; ++u, ++uc) {
          const PUnit U = load_punit(a, u);
          ok = wait(FP8 ? b_qready : b_qfull, uc & 1);   // FP8: hi and lo written in both CTAs
          for (int k = 0; k < U.te - U.tb && ok; ++k, ++n) {
            const uint32_t sb = n & 1, sph = (n >> 1) & 1;   // S^T buffer
            ok = wait(b_sempty + 8 * sb, sph ^ 1);
            const uint32_t d = tmem + sb * 128;
            if constexpr (FP8) {
              // the whole key tile: 9 chunks x 2 K steps, each K . hi then K . lo
              ok = ok && wait(b_ktfull, nkt & 1);
              if (!ok) break;
              tc_fence_after();
#pragma unroll
              for (int c = 0; c < 9; ++c) {
                const uint64_t bd = dQ0 + (uint64_t)(c * (q_chunk >> 4));
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                  const uint64_t ak = dKT0 + (uint64_t)(c * (512 >> 4) + 2 * kk);
                  umma_pair_f8(d, ak, bd + 2 * kk, idesc_qk, (c | kk) != 0);           // K . hi
                  umma_pair_f8(d, ak, bd + (512 >> 4) + 2 * kk, idesc_qk, 1u);         // K . lo
                }
              }
              umma_pair_commit(b_ktempty);
              ++nkt;
            }
            for (int ks = 0; !FP8 && ks < kKeySlots && ok; ++ks) {
              const int nc = 9 - KC * ks < KC ? 9 - KC * ks : KC;   // chunks KC ks .. (the last slot: 8)
              const uint32_t slot = r % kRing;
              ok = wait(b_full + 8 * slot, (r / kRing) & 1);
              if (!ok) break;
              tc_fence_after();
              const uint64_t ad = dK0 + (uint64_t)(slot * (kSlotBytes >> 4));
#pragma unroll
              for (int cc = 0; cc < KC; ++cc) {
                if (cc >= nc) break;
                const int c = KC * ks + cc;
                const uint64_t bd = dQ0 + (uint64_t)(c * (q_chunk >> 4));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  umma_pair_f16(d, ad + (uint64_t)(cc * (1024 >> 4) + 2 * kk), bd + 2 * kk, idesc_qk, (c | kk) != 0);
              }
              umma_pair_commit(b_empty + 8 * slot);
              ++r;
            }
            if (!ok) break;
            umma_pair_commit(b_sfull + 8 * sb);
            if (k == U.te - U.tb - 1) umma_pair_commit(b_qempty);
            if (prev.tile >= 0) ok = issue_pv(prev);
            prev = Prev{U.L, U.tb + k, k == 0, uc};
          }
          // the unit's last PV before the next unit's first QK^T: the epilogue waits for it,
          // while the next unit's QK^T can run during the epilogue
          if (ok && prev.tile >= 0) ok = issue_pv(prev);
          prev.tile = -1;
        }
        // every MMA issued has completed before tensor memory is released
        umma_pair_commit(b_drain);
        volatile uint32_t no_abort = 0;
        mbar_wait(b_drain, 0, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
      }
    } else if (FP8 && warp >= 2) {
      // ================================================================ Q converters (FP8)
      // Each unit's 64 query rows of this CTA, bf16 as TMA landed them, become q' = q 2^e (the
      // row's largest |q| in [128, 256)) written as E4M3 hi and lo in place: every 1 KB block
      // of 8 rows x 64 columns (128-byte swizzled bf16) becomes hi in its first 512 bytes and
      // lo in its second (8 rows x 64 bytes, 64-byte swizzled each), the QK^T MMAs' B operand.
      // A warp owns whole 8-row groups (all 9 blocks of them), so its reads of a group precede
      // its writes there; lane 4 q + p holds 16-byte units p and p + 4 of row q of each block.
      // The row factors 2^-e go to qf_s for the softmax warpgroup of these rows.
      constexpr uint32_t cbar = 3;                 // named barrier of the 64 converting threads
      const int qrow = lane >> 2, part = lane & 3;
      uint32_t uq = 0;
      for (int u = u0; u < u1; ++u, ++uq) {
        bool mine = wait(b_qraw, uq & 1);
        if (mine && uq > 0) mine = wait(b_qfree, (uq - 1) & 1);   // the previous factors were read
        if (named_bar_or(cbar, 64, !mine)) break;
        for (int g = warp - 2; g < 8; g += 2) {
          auto block_of = [&](int c) -> uint8_t* {
            return gQ + (a.q_whole_rows ? g * 9216 + c * 1024 : c * kQChunk + g * 1024);
          };
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
              for (int k = 0; k < 4; ++k) o[k] = split_e4m3x2(bf16_lo(w[k]) * f, bf16_hi(w[k]) * f);
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
        named_bar_sync(cbar, 64);
        if (threadIdx.x == 64) {
          mbar_arrive(b_qsc);
          // the even CTA's MMA issuer needs both CTAs' Q: the odd CTA signals by st.async
          if (leader) mbar_arrive_expect_tx(b_qready, 16);
          else st_async_v4(lead(smem_u32(sig_s)), make_uint4(0u, 0u, 0u, 0u), lead(b_qready));
        }
      }
    }
  } else if (warp >= 4) {
    // ================================================================ softmax / epilogue
    const int wg = (warp - 4) >> 2;                // rows 64 wg .. 64 wg + 63
    const int wl = warp & 3;                       // TMEM lane quarter
    const int t = wl * 32 + lane;                  // key of this CTA's half of the tile
    const uint32_t bar = 1 + wg;
    const uint32_t lane_addr = (uint32_t)(wl * 32) << 16;
    const bool local_p = (uint32_t)wg == rank;     // this warpgroup's rows live in this CTA
    const float kvs = FP8 ? __ldg(a.kv_scale) : 1.0f;
    const float c_log2 = a.softmax_scale * kvs * kPLog2e;
    const float kvo = kvs;
    float* mref = mref_s[wg];
    const float* rowc = rowc_s[wg];
    uint32_t gn = 0, xc = 0;
    bool ok = true;
    auto wait_wg = [&](uint32_t b, uint32_t parity) -> bool { return !named_bar_or(bar, 128, !wait(b, parity)); };
    // One exchange with the same warpgroup of the peer CTA: a 272-byte message (a flag and
    // 64 values) sent with st.async, its bytes counted on the peer's barrier, which the peer
    // arms itself; every thread then waits for the peer's message.
    auto exchange = [&](uint32_t flag, const float* vals) -> const float* {
      const uint32_t par = xc & 1, xb = b_x + 8 * (2 * wg + par);
      named_bar_sync(bar, 128);                    // vals complete
      if (t == 0) mbar_arrive_expect_tx(xb, 272);
      if (t < 17) {
        const uint32_t dst = map_to_rank(smem_u32(&xbuf[wg][par][0]), peer) + 16 * t;
        const uint4 v = t == 0 ? make_uint4(flag, 0, 0, 0) : *reinterpret_cast<const uint4*>(vals + 4 * (t - 1));
        st_async_v4(dst, v, map_to_rank(xb, peer));
      }
      const bool w = mbar_wait_cluster(xb, (xc >> 1) & 1, abort_flag, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
      ++xc;
      if (named_bar_or(bar, 128, !w)) {
        if (t == 0) fail_peer();
        return nullptr;
      }
      return &xbuf[wg][par][0];
    };
    // Sum of v over the 32 lanes for 64 rows at once (reduce-scatter): afterwards lane l
    // holds the sums of rows 2l and 2l + 1 in v[0], v[1].
    auto reduce_rows = [&](float* v) {
#pragma unroll
      for (int n = 64, off = 16; off > 0; n >>= 1, off >>= 1) {
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const float keep = hi ? v[i + n / 2] : v[i];
          const float send = hi ? v[i] : v[i + n / 2];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
    };

    // The same with max over the rows of v, which is left unchanged: lane l gets the maxima of
    // rows 2l and 2l + 1.
    auto reduce_rows_max = [&](const float* v, float& m0, float& m1) {
      float w[32];
      {
        const bool hi = (lane & 16) != 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float keep = hi ? v[i + 32] : v[i];
          const float send = hi ? v[i] : v[i + 32];
          w[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
        }
      }
#pragma unroll
      for (int n = 32, off = 8; off > 0; n >>= 1, off >>= 1) {
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const float keep = hi ? w[i + n / 2] : w[i];
          const float send = hi ? w[i] : w[i + n / 2];
          w[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, off));
        }
      }
      m0 = w[0];
      m1 = w[1];
    };

    float lsum[64];
    for (int u = u0; u < u1 && ok; ++u) {
      const uint32_t ui = (uint32_t)(u - u0);     // this CTA's unit count
      const PUnit U = load_punit(a, u);
      const int T = U.te - U.tb;
      const int row0 = U.g * 128 + 64 * wg;        // first row of this warpgroup in the sequence
      if (t < 64) {
        mref[t] = -INFINITY;
        nvis_s[wg][t] = a.causal ? min(U.L, U.L - a.s_q + 1 + (row0 + t) / a.H) : U.L;
      }
      if constexpr (FP8) {
        // the unit's row factors 2^-e: from this CTA's converters for the warpgroup whose rows
        // live here, which passes them to the same warpgroup of the peer
        if (local_p) {
          ok = wait_wg(b_qsc, ui & 1);
          if (!ok) break;
          if (t < 64) own_s[wg][t] = qf_s[t];
        }
        const float* px = exchange(0u, own_s[wg]);
        if (px == nullptr) { ok = false; break; }
        if (local_p && t == 0) mbar_arrive(b_qfree);
        if (t < 64) rowc_s[wg][t] = c_log2 * (local_p ? own_s[wg][t] : px[4 + t]);
      }
      const int mask_from = a.causal ? U.L - a.s_q + 1 : U.L;
#pragma unroll
      for (int i = 0; i < 64; ++i) lsum[i] = 0.f;
      named_bar_sync(bar, 128);
      for (int k = 0; k < T && ok; ++k) {
        const uint32_t n = gn + k;
        const int tile = U.tb + k;
        if (a.test_stall && n == 0) {
          ok = wait_wg(b_never, 0);                  // tests: this wait runs out
          if (!ok) break;
        }
        const uint32_t sb = n & 1, sph = (n >> 1) & 1;   // S^T buffer
        ok = wait_wg(b_sfull + 8 * sb, sph);
        if (!ok) break;
        tc_fence_after();
        float s[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16(tmem + lane_addr + sb * 128 + 64 * wg + 16 * c, s + 16 * c);
        tmem_wait_ld();
        tc_fence_before();

        const int j = tile * kPairKeys + 128 * (int)rank + t;
        bool need = false;
        // the score factor of 4 rows: bf16 one constant, FP8 per row (2^-e of its q)
        auto factors = [&](int r, float* cc) {
          if constexpr (FP8) {
            const float4 c4 = *reinterpret_cast<const float4*>(rowc + r);
            cc[0] = c4.x; cc[1] = c4.y; cc[2] = c4.z; cc[3] = c4.w;
          } else {
            cc[0] = cc[1] = cc[2] = cc[3] = c_log2;
          }
        };
        if ((tile + 1) * kPairKeys <= mask_from) {
#pragma unroll
          for (int r = 0; r < 64; r += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mref + r);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
            float cc[4];
            factors(r, cc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              s[r + i] *= cc[i];
              need |= s[r + i] > mm[i] + Cfg::kRescaleLog2;
            }
          }
        } else {
#pragma unroll
          for (int r = 0; r < 64; r += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mref + r);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
            float cc[4];
            factors(r, cc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              s[r + i] = j < nvis_s[wg][r + i] ? s[r + i] * cc[i] : -INFINITY;
              need |= s[r + i] > mm[i] + Cfg::kRescaleLog2;
            }
          }
        }
        // the barrier also orders every thread's S^T reads before the even CTA's signal; the
        // odd CTA's S^T reads precede its P^T signal, which the MMA issuer awaits before it
        // reuses the buffer two tiles later
        const bool need_local = named_bar_or(bar, 128, need);
        if (leader && t == 0) mbar_arrive(b_sempty + 8 * sb);
        if (need_local) {
          // column maxima of the warp's 32 keys for all 64 rows at once (reduce-scatter,
          // as for the row sums)
          float m0, m1;
          reduce_rows_max(s, m0, m1);
          wred_s[wg][wl][2 * lane] = m0;
          wred_s[wg][wl][2 * lane + 1] = m1;
          named_bar_sync(bar, 128);
          if (t < 64)
            own_s[wg][t] = fmaxf(fmaxf(wred_s[wg][0][t], wred_s[wg][1][t]), fmaxf(wred_s[wg][2][t], wred_s[wg][3][t]));
        }
        const float* px = exchange(need_local ? 1u : 0u, own_s[wg]);
        if (px == nullptr) { ok = false; break; }
        const bool need_peer = __float_as_uint(px[0]) != 0u;
        bool rescale = false;
        if (need_local || need_peer) {
          if (t < 64) {
            const float old = mref[t];
            float nm = old;
            if (need_local) nm = fmaxf(nm, own_s[wg][t]);
            if (need_peer) nm = fmaxf(nm, px[4 + t]);
            alpha_s[wg][t] = nm == -INFINITY ? 1.f : ex2_approx(old - nm);
            mref[t] = nm;
          }
          named_bar_sync(bar, 128);
#pragma unroll
          for (int r = 0; r < 64; ++r) lsum[r] *= alpha_s[wg][r];
          rescale = k > 0;
        }
        // bf16: 32 words of P^T pairs. FP8: P times 2^4, its hi bytes (words 0-15) and lo
        // bytes (words 16-31), four rows per word
        uint32_t pw[32];
#pragma unroll
        for (int r = 0; r < 64; r += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(mref + r);
          const float mm[4] = {m4.x - Cfg::kPOffLog2, m4.y - Cfg::kPOffLog2, m4.z - Cfg::kPOffLog2,
                               m4.w - Cfg::kPOffLog2};
          float p[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            p[i] = s[r + i] == -INFINITY ? 0.f : ex2_approx(s[r + i] - mm[i]);
            lsum[r + i] += p[i];                 // the normaliser sums the unrounded values
          }
          if constexpr (FP8) {
            const uint32_t o0 = split_e4m3x2(p[0], p[1]), o1 = split_e4m3x2(p[2], p[3]);
            pw[r / 4] = __byte_perm(o0, o1, 0x5410);
            pw[16 + r / 4] = __byte_perm(o0, o1, 0x7632);
          } else {
            __nv_bfloat162 h0 = __floats2bfloat162_rn(p[0], p[1]), h1 = __floats2bfloat162_rn(p[2], p[3]);
            pw[r / 2] = *reinterpret_cast<uint32_t*>(&h0);
            pw[r / 2 + 1] = *reinterpret_cast<uint32_t*>(&h1);
          }
        }
        // P^T and O^T are free once the previous PV has completed; the staging buffer once
        // the previous copy out of it has been read
        if (!FP8 && t == 0 && !local_p) bulk_wait_read0();
        if (n > 0) {
          ok = wait_wg(b_pvdone, (n - 1) & 1);
          if (!ok) break;
        } else {
          named_bar_sync(bar, 128);
        }
        if (rescale) {
          tc_fence_after();
#pragma unroll 1
          for (int jt = 0; jt < 2; ++jt) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              float o[16];
              const uint32_t ta = tmem + lane_addr + kOCol + 128 * jt + 64 * wg + 16 * c;
              tmem_ld16(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= alpha_s[wg][16 * c + i];
              tmem_st16(ta, o);
            }
          }
          tmem_wait_st();
        }
        // P^T row of key 128 rank + t: into this CTA's P^T buffer (rows 64 rank ..), or, for
        // the peer: bf16 into the staging buffer laid out as the peer's P^T rows of keys
        // 128 rank .. 128 rank + 127 (sent by one bulk copy below); FP8 straight into the
        // peer's P^T by st.async, its bytes counted on the peer's barrier
        if constexpr (FP8) {
          const uint32_t pdst = local_p ? sP + (uint32_t)rank * kStageBytes
                                        : map_to_rank(sP + (uint32_t)rank * kStageBytes, peer);
          const uint32_t pbar = map_to_rank(leader ? b_pin : b_pfull, peer);
#pragma unroll
          for (int hl = 0; hl < 2; ++hl)
#pragma unroll
            for (int u16 = 0; u16 < 4; ++u16) {
              const uint32_t off = hl * 8192 + p_off64(t, u16);
              const uint4 v = make_uint4(pw[16 * hl + 4 * u16], pw[16 * hl + 4 * u16 + 1], pw[16 * hl + 4 * u16 + 2],
                                         pw[16 * hl + 4 * u16 + 3]);
              if (local_p) *reinterpret_cast<uint4*>(gP + (pdst - sP) + off) = v;
              else st_async_v4(pdst + off, v, pbar);
            }
        } else {
          uint8_t* prow = local_p ? gP + (int)rank * kStageBytes : gStage;
#pragma unroll
          for (int u16 = 0; u16 < 8; ++u16)
            *reinterpret_cast<uint4*>(prow + p_off128(t, u16)) =
                make_uint4(pw[4 * u16], pw[4 * u16 + 1], pw[4 * u16 + 2], pw[4 * u16 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(bar, 128);
        if (t == 0) {
          if (!local_p) {
            // bf16: the rows for the peer's P^T in one bulk copy, counted on the peer's barrier
            // (the even CTA's P^T barrier, or the odd CTA's b_pin); FP8: already sent
            if (!FP8) {
              bulk_copy_to_cluster(map_to_rank(sP + (uint32_t)rank * kStageBytes, peer), sStage, kStageBytes,
                                   map_to_rank(leader ? b_pin : b_pfull, peer));
              bulk_commit();
            }
          } else if (leader) {
            mbar_arrive_expect_tx(b_pfull, kStageBytes);   // own rows; the odd CTA's rows to come
          } else {
            mbar_arrive_expect_tx(b_pin, kStageBytes);
            ok = mbar_wait(b_pin, n & 1, abort_flag, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);   // the even CTA's rows
            if (FP8 && ok) fence_proxy_async_smem();   // rows that came by st.async, for the MMAs
            if (ok) mbar_arrive_cluster(lead(b_pfull));
            else fail_peer();
          }
        }
        if (!local_p || leader) continue;
        ok = !named_bar_or(bar, 128, !ok);
      }
      if (!ok) break;
      // ---- epilogue: the unit's last PV, row sums of both CTAs, O^T / l -> output
      ok = wait_wg(b_pvdone, (gn + T - 1) & 1);
      if (!ok) break;
      tc_fence_after();
      reduce_rows(lsum);
      wred_s[wg][wl][2 * lane] = lsum[0];
      wred_s[wg][wl][2 * lane + 1] = lsum[1];
      named_bar_sync(bar, 128);
      if (t < 64) own_s[wg][t] = (wred_s[wg][0][t] + wred_s[wg][1][t]) + (wred_s[wg][2][t] + wred_s[wg][3][t]);
      const float* px = exchange(1u, own_s[wg]);
      if (px == nullptr) { ok = false; break; }
      float tot = 0.f;
      if (t < 64) {
        tot = own_s[wg][t] + px[4 + t];           // addition commutes: the same in both CTAs
        alpha_s[wg][t] = tot > 0.f ? kvo / tot : 0.f;
      }
      named_bar_sync(bar, 128);
      const bool direct = U.slot < 0;
      // Each warp holds value columns 256 rank + 128 jt + 32 wl + lane (its TMEM lanes) of 16
      // rows per load. Each quad of lanes transposes 4 x 4 blocks of them in registers (two
      // shuffle steps), after which lane 4q + j holds row j of a block at 4 consecutive
      // columns: 8-byte (bf16 output) or 16-byte (float32 partial) stores, and no shared
      // memory traffic next to the MMAs of the next unit.
      const int nrows = min(64, R - row0);         // rows of this warpgroup that exist
      const int qj = lane & 3;
#pragma unroll 1
      for (int jt = 0; jt < 2; ++jt) {
        // the warpgroup's 64 rows of these 128 value columns, in one batch of loads
        float ob[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16(tmem + lane_addr + kOCol + 128 * jt + 64 * wg + 16 * c, ob + 16 * c);
        tmem_wait_ld();
        if (jt == 1) {
          // O^T has been read: the next unit's first PV may overwrite it
          tc_fence_before();
          named_bar_sync(bar, 128);
          if (leader && t == 0) mbar_arrive(b_oempty);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float* o = ob + 16 * c;
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= alpha_s[wg][16 * c + i];
          const int col = 256 * (int)rank + 128 * jt + 32 * wl + 4 * (lane >> 2);
          if (direct) {
#pragma unroll
            for (int bp = 0; bp < 2; ++bp) {
              // rows 8 bp + i (low halves) and 8 bp + 4 + i (high halves) as bf16 pairs
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                __nv_bfloat162 h = __floats2bfloat162_rn(o[8 * bp + i], o[8 * bp + 4 + i]);
                w[i] = *reinterpret_cast<uint32_t*>(&h);
              }
              quad_transpose4(w, qj);
              const int r0 = 16 * c + 8 * bp + qj;   // rows r0 (low halves) and r0 + 4 (high)
              if (r0 < nrows)
                *reinterpret_cast<uint2*>(a.out + ((int64_t)U.b * R + row0 + r0) * kDV + col) =
                    make_uint2(__byte_perm(w[0], w[1], 0x5410), __byte_perm(w[2], w[3], 0x5410));
              if (r0 + 4 < nrows)
                *reinterpret_cast<uint2*>(a.out + ((int64_t)U.b * R + row0 + r0 + 4) * kDV + col) =
                    make_uint2(__byte_perm(w[0], w[1], 0x7632), __byte_perm(w[2], w[3], 0x7632));
            }
          } else {
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) w[i] = __float_as_uint(o[4 * blk + i]);
              quad_transpose4(w, qj);
              const int r = 16 * c + 4 * blk + qj;   // row 64 wg + r of the unit
              if (r < nrows)
                *reinterpret_cast<float4*>(a.part_o + ((int64_t)U.slot * 128 + 64 * wg + r) * kDV + col) =
                    make_float4(__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]),
                                __uint_as_float(w[3]));
            }
          }
        }
      }
      if (rank == 0 && t < 64 && row0 + t < R) {
        // P was computed times 2^kPOffLog2, and so was the row sum
        const float l = tot > 0.f ? (mref[t] + __log2f(tot) - Cfg::kPOffLog2) * kPLn2 : -INFINITY;
        if (direct) a.lse[(int64_t)U.b * R + row0 + t] = l;
        else a.part_lse[(int64_t)U.slot * 128 + 64 * wg + t] = l;
      }
      named_bar_sync(bar, 128);
      gn += T;
    }
    // a copy out of the staging buffer has landed before the CTA may leave
    if (!FP8 && t == 0 && !local_p) bulk_wait0();
  }

  // ================================================================ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();                         // neither CTA leaves while its peer may still use it
  tc_fence_after();
  if (warp == 0) tmem_dealloc_pair(tmem, kPairTmemCols);
}

template <bool FP8, bool kSub>
static cudaError_t prepare_pair_variant() {
  cudaError_t e = cudaFuncSetAttribute(decode_pair_kernel<FP8, kSub>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       pair_dyn_bytes(FP8));
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, decode_pair_kernel<FP8, kSub>);
  if (e != cudaSuccess) return e;
  if ((int)attr.sharedSizeBytes > kPairStaticBudget) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

template <bool FP8>
static cudaError_t launch_pair_variant(const DecodeArgs& a, int pairs, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = pair_dyn_bytes(FP8);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the scheduler
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // pages smaller than 64 rows take the kernel that loads a 64-key block as several boxes
  return a.box_rows < 64 ? cudaLaunchKernelEx(&cfg, decode_pair_kernel<FP8, true>, a)
                         : cudaLaunchKernelEx(&cfg, decode_pair_kernel<FP8, false>, a);
}

cudaError_t decode_pair_prepare(bool fp8) {
  cudaError_t e = fp8 ? prepare_pair_variant<true, false>() : prepare_pair_variant<false, false>();
  if (e != cudaSuccess) return e;
  return fp8 ? prepare_pair_variant<true, true>() : prepare_pair_variant<false, true>();
}

cudaError_t launch_decode_pair(const DecodeArgs& a, bool fp8, int pairs, cudaStream_t s) {
  if (pairs < 1) return cudaErrorInvalidValue;
  return fp8 ? launch_pair_variant<true>(a, pairs, s) : launch_pair_variant<false>(a, pairs, s);
}

}  // namespace mla
