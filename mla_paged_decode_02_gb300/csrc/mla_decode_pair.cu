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
// Softmax coupling. Both CTAs' keys accumulate into the same O^T rows, so they share one
// reference maximum per row. Each CTA runs two softmax warpgroups, warpgroup w for rows
// 64w..64w+63 (one thread per key = one TMEM lane). Per tile the warpgroup tells the
// same warpgroup of the peer whether any of its scores exceeds the reference by more than
// 2^8 (and, only then, its row maxima) through distributed shared memory; both then move
// the reference identically. P^T rows 64w.. go to CTA w's P^T buffer (its own or the
// peer's shared memory). At the end of a unit the row sums are exchanged the same way.
//
// Pipeline per CTA (384 threads). Warp 0: producer — one ring of 32 KB slots in the order
// the MMAs consume them (the 5 key slots of tile n, then the value slots of tile n-1; a
// unit's last value slots right after its last key slots), plus each unit's Q. A TMA load's cost grows with the number of contiguous row pieces in its
// box (measured on this GPU: about 22 GB/s per SM for 128-byte pieces from L2, 44 for 256,
// 87 for 512), so key boxes take two adjacent 64-column chunks of each row and value boxes
// four. Every load completes on the even CTA's barrier, which the even CTA alone arms with
// the bytes of both CTAs (it knows which key halves its peer loads), so that no load needs a
// cross-CTA arrival (each costs a fraction of a microsecond). Warp 1 of the even CTA: the
// single MMA issuer, in program order QK^T(n), PV(n-1), QK^T(n+1), ..., a unit's last PV
// before the next unit's first QK^T (so that the epilogue need not wait for it); its commits arrive
// on the barrier at the same offset in both CTAs. Warps 4-7 and 8-11: softmax warpgroups 0
// and 1, then the epilogue. Every wait is bounded; a stall sets the device error word, and
// both CTAs drain and leave through a final cluster barrier.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "mla_internal.h"
#include "mla_pages.cuh"
#include "mla_ptx.cuh"
#include "../../include/mla.h"

namespace mla {
namespace {

constexpr int kPairKeys = 256;              // keys per super-tile
constexpr int kSlotBytes = 32768;           // ring slot: 128 keys x 128 columns, or 64 keys x 256 columns
constexpr int kKeySlots = 5;                // key chunk pairs per super-tile (9 chunks, the last alone)
constexpr int kQChunk = 8192;               // 64 rows x 64 columns bf16
constexpr int kPairQBytes = 9 * kQChunk;
constexpr int kPairPBytes = kPairKeys * 128;  // P^T: 256 keys x 64 rows bf16
constexpr int kStageBytes = 16384;         // P^T rows bound for the peer: 128 keys x 64 rows
constexpr int kRawSlotBytes = 16384;       // FP8 raw slot: 128 keys x 2 chunks, or 64 keys x 4 chunks, E4M3
constexpr int kMaxRing = 3;
constexpr int kPairTmemCols = 512;
constexpr int kOCol = 256;                  // O^T M-tile j at columns 256 + 128 j
constexpr float kPairRescaleLog2 = 8.0f;
constexpr float kPLog2e = 1.4426950408889634f;
constexpr float kPLn2 = 0.6931471805599453f;
constexpr int kPairSmemLimit = 232448;
constexpr int kPairStaticBudget = 9216;

// bf16: 384 threads; a ring of three 32 KB operand slots (keys and values) filled by TMA,
// and a 16 KB staging buffer for the P^T rows sent to the peer by one bulk copy; S^T
// double-buffered in tensor memory.
// FP8: 512 threads (a fourth warpgroup converts E4M3 to fp16); keys go to two tensor-memory
// key slots (the QK^T MMAs read A from tensor memory), values to a ring of two 32 KB fp16
// slots, both from a ring of three 16 KB raw E4M3 slots filled by TMA; S^T single-buffered
// (its second buffer's columns hold the key slots); P^T rows for the peer go by st.async
// (no staging buffer).
template <bool FP8>
struct PairCfg {
  static constexpr int kThreads = FP8 ? 512 : 384;
  static constexpr int kRing = FP8 ? 2 : 3;
  static constexpr int kStage = FP8 ? 0 : kStageBytes;
  static constexpr int kRawRing = FP8 ? 3 : 0;
  static constexpr int kDynBytes =
      1024 + kPairQBytes + kPairPBytes + kStage + kRing * kSlotBytes + kRawRing * kRawSlotBytes;
  static_assert(kRing <= kMaxRing && kRawRing <= kMaxRing, "barrier arrays");
  static_assert(kDynBytes + kPairStaticBudget <= kPairSmemLimit, "shared memory budget");
};
constexpr int kKeyTSlots = 2;               // FP8: tensor-memory key slots (two chunks = 64 columns each)
constexpr int kKeyCol = 128;                // FP8: their first column
// FP8 register budgets per thread (setmaxnreg): warpgroup 0 (producer, MMA issuer), the two
// softmax warpgroups, the converters. They redistribute the launch allocation of 128.
constexpr int kRegsCtl = 96, kRegsSoftmax = 176, kRegsConv = 64;
static_assert(kRegsCtl + 2 * kRegsSoftmax + kRegsConv <= 4 * 128, "register budgets exceed the launch allocation");

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

__device__ __forceinline__ uint32_t p_off128(int row, int u) {   // 128-byte swizzled P^T row
  return (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u + ((uint32_t)(u ^ (row & 7)) << 4);
}

}  // namespace

template <bool FP8, bool kSub>
__global__ void __launch_bounds__(PairCfg<FP8>::kThreads, 1) decode_pair_kernel(const __grid_constant__ DecodeArgs a) {
  using Cfg = PairCfg<FP8>;
  // (the raw ring's depth is 1, not 0, in the bf16 kernel, where no code indexes it)
  constexpr int kRing = Cfg::kRing, kRawRing = FP8 ? Cfg::kRawRing : 1;
  extern __shared__ uint8_t dsmem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kMaxRing], bar_empty[kMaxRing], bar_aux;
  __shared__ __align__(8) uint64_t bar_qfull, bar_qempty;
  // FP8: raw ring, Q landed (this CTA), Q converted (both CTAs, on the even CTA)
  __shared__ __align__(8) uint64_t bar_rfull[kMaxRing], bar_rempty[kMaxRing], bar_qraw, bar_qready;
  __shared__ __align__(8) uint64_t bar_kfull[kKeyTSlots], bar_kempty[kKeyTSlots];   // FP8 key slots
  __shared__ __align__(16) uint32_t sig_s[4];        // landing place of the odd CTA's 16-byte signals
  __shared__ __align__(8) uint64_t bar_sfull[2], bar_sempty[2], bar_pfull, bar_pin, bar_pvdone, bar_oempty;
  __shared__ __align__(8) uint64_t bar_x[2][2];
  __shared__ __align__(8) uint64_t bar_drain, bar_never, bar_epi;
  __shared__ uint32_t tmem_base_s, abort_s;
  __shared__ __align__(16) float xbuf[2][2][68];     // [warpgroup][parity]: word 0 flag, words 4..67 values
  __shared__ __align__(16) float mref_s[2][64];
  __shared__ float alpha_s[2][64], own_s[2][64];
  __shared__ int nvis_s[2][64];
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
  const uint32_t sStage = sP + kPairPBytes;
  const uint32_t sR = sStage + Cfg::kStage;
  const uint32_t sRaw = sR + kRing * kSlotBytes;     // FP8 raw ring
  uint8_t* gQ = gbase;
  uint8_t* gP = gbase + kPairQBytes;
  uint8_t* gStage = gP + kPairPBytes;
  uint8_t* gR = gStage + Cfg::kStage;
  const uint8_t* gRaw = gR + kRing * kSlotBytes;

  const uint32_t b_full = smem_u32(bar_full), b_empty = smem_u32(bar_empty), b_aux = smem_u32(&bar_aux);
  const uint32_t b_qfull = smem_u32(&bar_qfull), b_qempty = smem_u32(&bar_qempty);
  const uint32_t b_sfull = smem_u32(bar_sfull), b_sempty = smem_u32(bar_sempty);
  const uint32_t b_pfull = smem_u32(&bar_pfull), b_pin = smem_u32(&bar_pin), b_pvdone = smem_u32(&bar_pvdone);
  const uint32_t b_oempty = smem_u32(&bar_oempty), b_drain = smem_u32(&bar_drain);
  const uint32_t b_x = smem_u32(bar_x);
  const uint32_t b_never = smem_u32(&bar_never);   // tests: a barrier nothing arrives on
  const uint32_t b_epi = smem_u32(&bar_epi);       // FP8: a unit's epilogue scratch is free again
  const uint32_t b_rfull = smem_u32(bar_rfull), b_rempty = smem_u32(bar_rempty);
  const uint32_t b_qraw = smem_u32(&bar_qraw), b_qready = smem_u32(&bar_qready);
  const uint32_t b_kfull = smem_u32(bar_kfull), b_kempty = smem_u32(bar_kempty);
  volatile uint32_t* abort_flag = &abort_s;
  uint32_t* err = a.err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      // bf16: the even CTA's producer, with both CTAs' bytes; FP8: the even CTA's
      // converters, expecting the odd CTA's converters' 16-byte message
      mbar_init(b_full + 8 * i, 1);
      mbar_init(b_empty + 8 * i, 1);
    }
    for (int i = 0; i < Cfg::kRawRing; ++i) {
      mbar_init(b_rfull + 8 * i, 1);      // this CTA's producer, with its bytes
      mbar_init(b_rempty + 8 * i, 1);     // this CTA's converters
    }
    mbar_init(b_qraw, 1);
    mbar_init(b_qready, 1);               // as b_full (FP8)
    for (int i = 0; i < kKeyTSlots; ++i) {
      mbar_init(b_kfull + 8 * i, 1);      // as b_full (FP8)
      mbar_init(b_kempty + 8 * i, 1);
    }
    mbar_init(b_aux, 1);
    mbar_init(b_qfull, 1);                // the even CTA's arrival, with both CTAs' bytes
    mbar_init(b_qempty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_sfull + 8 * i, 1);
      // the even CTA's two warpgroups (bf16: the odd CTA's reads precede its P^T signals;
      // FP8: each expects 16 bytes from the odd CTA's warpgroup of the same rows)
      mbar_init(b_sempty + 8 * i, 2);
    }
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
    mbar_init(b_epi, 1);                  // FP8: the warpgroup whose P^T rows live in the peer
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
  // arrive on a barrier of the even CTA (a local arrive there, a remote one from the odd CTA)
  auto arrive_lead = [&](uint32_t addr) {
    if (leader) mbar_arrive(addr);
    else mbar_arrive_cluster(lead(addr));
  };
  // A failed wait also raises the peer's abort flag, so that its waits end too.
  auto fail_peer = [&]() { st_cluster_u32(map_to_rank(smem_u32(&abort_s), peer), 1u); };
  auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = mbar_wait(bar, parity, abort_flag, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
    if (!ok) fail_peer();
    return ok;
  };

  if (warp < 4) {
    // warpgroup 0: producer (warp 0) and MMA issuer (warp 1 of the even CTA). FP8: every
    // warpgroup first sets its register budget (all four warps, before they split).
    if constexpr (FP8) regs_lower<kRegsCtl>();
    if (warp == 0) {
      if constexpr (FP8) {
      // ================================================================ producer (FP8)
      // Raw E4M3 rows into this CTA's raw ring in the order the converters (and then the
      // MMAs) take them — per super-tile its 5 key slots, then the value slots of the
      // previous one, a unit's last value slots right after its last key slots — and each
      // unit's Q. Every load completes on this CTA's own barrier: only the converters' output
      // is shared with the peer.
      uint32_t rr = 0, uq = 0;
      bool ok = true;
      const uint64_t pol_keep = l2_policy_evict_last(), pol_last = l2_policy_evict_first();
      const int32_t* bt_all = a.block_table;
      const uint32_t box_rows = kSub ? (uint32_t)a.box_rows : 64u;
      const uint32_t kbox_bytes = 128 * box_rows;        // raw key box: 2 chunks x 64 B per row
      const uint32_t vbox_bytes = 256 * box_rows;        // raw value box: 4 chunks x 64 B per row
      // the next raw slot once the converters have released it (-1: a wait gave up)
      auto take_raw = [&]() -> int {
        const uint32_t rs = rr % kRawRing;
        const bool w_ok = lane != 0 || wait(b_rempty + 8 * rs, ((rr / kRawRing) & 1) ^ 1);
        return __all_sync(0xffffffffu, w_ok) ? (int)rs : -1;
      };
      // raw value slot [8 key groups][4 chunks][8 rows][64 B]: this CTA's value columns of
      // one 64-key block (rows past the sequence end are zeroed by the converters)
      auto load_values = [&](const PUnit& U, int tile, const int64_t* rb, const int* nb) -> bool {
        const int32_t* bt = bt_all + (int64_t)U.b * a.MB;
        for (int kb = 0; kb < 4; ++kb) {
          if (rb[kb] < 0) continue;
          const int rs = take_raw();
          if (rs < 0) return false;
          if (lane == 0) {
            const uint32_t bar = b_rfull + 8 * rs, dst = sRaw + rs * kRawSlotBytes;
            const int32_t c0 = 4 * (int)rank;            // this CTA's value columns 256 rank ..
            mbar_arrive_expect_tx(bar, (kSub ? (uint32_t)nb[kb] : 1u) * vbox_bytes);
            tma_load_4d_hint(dst, &a.tm_v, bar, 0, 0, c0, (int32_t)(rb[kb] >> 3), pol_last);
            if (kSub && nb[kb] > 1)
              load_more_boxes(kBoxHint, &a.tm_v, dst, bar, c0, vbox_bytes, bt, a, tile * kPairKeys + 64 * kb, nb[kb],
                              pol_last);
          }
          ++rr;
        }
        return true;
      };
      PUnit pu{};
      int ptile = -1;
      int64_t prb[4] = {-1, -1, -1, -1};
      int pnb[4] = {0, 0, 0, 0};
      for (int u = u0; u < u1 && ok; ++u, ++uq) {
        const PUnit U = load_punit(a, u);
        // this CTA's 64 query rows (bf16; the converters turn them into fp16 in place) once
        // the previous unit's QK^T MMAs are done with the buffer
        bool w_ok = lane != 0 || wait(b_qempty, (uq & 1) ^ 1);
        ok = __all_sync(0xffffffffu, w_ok);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(b_qraw, kPairQBytes);
          if (a.q_whole_rows)
            tma_load_5d_hint(sQ, &a.tm_q, b_qraw, 0, 0, 0, (128 * U.g + 64 * (int)rank) / 8, U.b, pol_keep);
          else
            for (int c = 0; c < 9; ++c)
              tma_load_3d_hint(sQ + c * kQChunk, &a.tm_q, b_qraw, 64 * c, 128 * U.g + 64 * (int)rank, U.b, pol_keep);
        }
        for (int tile = U.tb; tile < U.te && ok; ++tile) {
          int64_t rb[4];
          int nb[4];
          block_rows<kSub>(a, U, tile, rb, nb);
          const int32_t* bt = bt_all + (int64_t)U.b * a.MB;
          const uint32_t nown = (uint32_t)(nb[2 * rank] + nb[2 * rank + 1]);   // this CTA's key boxes
          // raw key slot [2 halves][8 groups][2 chunks][8 rows][64 B]: chunks 2ks, 2ks + 1 of
          // this CTA's 128 keys (the last slot: chunk 8 and a zero-filled chunk past the row)
          for (int ks = 0; ks < kKeySlots; ++ks) {
            const int rs = take_raw();
            if (rs < 0) { ok = false; break; }
            if (lane == 0) {
              const uint32_t bar = b_rfull + 8 * rs, dst = sRaw + rs * kRawSlotBytes;
              mbar_arrive_expect_tx(bar, nown * kbox_bytes);
              for (int h = 0; h < 2; ++h) {
                const int kb = 2 * (int)rank + h;
                if (nb[kb] == 0) continue;
                const uint32_t d = dst + h * (kRawSlotBytes / 2);
                tma_load_4d_hint(d, &a.tm_k, bar, 0, 0, 2 * ks, (int32_t)(rb[kb] >> 3), pol_keep);
                if (kSub && nb[kb] > 1)
                  load_more_boxes(kBoxHint, &a.tm_k, d, bar, 2 * ks, kbox_bytes, bt, a, tile * kPairKeys + 64 * kb,
                                  nb[kb], pol_keep);
              }
            }
            ++rr;
          }
          if (!ok) break;
          if (ptile >= 0) ok = load_values(pu, ptile, prb, pnb);
          pu = U;
          ptile = tile;
          for (int kb = 0; kb < 4; ++kb) { prb[kb] = rb[kb]; pnb[kb] = nb[kb]; }
        }
        if (ok && ptile >= 0) ok = load_values(pu, ptile, prb, pnb);
        ptile = -1;
      }
      // this CTA's own loads have landed before it may leave
      if (lane == 0) {
        volatile uint32_t no_abort = 0;
        for (uint32_t q = rr > (uint32_t)kRawRing ? rr - kRawRing : 0; q < rr; ++q)
          mbar_wait(b_rfull + 8 * (q % kRawRing), (q / kRawRing) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT,
                    a.wait_limit_ns);
        if (uq > 0) mbar_wait(b_qraw, (uq - 1) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
      }
      } else {
      // ================================================================ producer
      // Ring order per super-tile n: its 5 key slots (chunk pairs 0-1, 2-3, 4-5, 6-7 and 8,
      // 128 keys each), then the value slots of tile n-1 (64 keys x this CTA's 256 value
      // columns each, one per 64-key block before the sequence end); a unit's last value
      // slots follow its last key slots. TMA cost grows with the number of contiguous row pieces a box has, not
      // with its bytes, so every box takes 2 (keys) or 4 (values) adjacent chunks of a row.
      uint32_t r = 0, uq = 0, aux = 0;
      bool ok = true;
      // a key's lines are read again (as values, by this CTA or its peer) about one tile later:
      // keep them in L2; the value read is their last use
      const uint64_t pol_keep = l2_policy_evict_last(), pol_last = l2_policy_evict_first();
      // the block holding the sequence end gets the rows up to the end of its last 16-key MMA
      // step zeroed (the cache may hold NaN there, and 0 * NaN is NaN inside the MMA)
      const int32_t* bt_all = a.block_table;
      const uint32_t box_rows = kSub ? (uint32_t)a.box_rows : 64u;             // rows of one box
      const uint32_t kbox_bytes = (kSlotBytes / 128) * box_rows;               // one key box
      const uint32_t vbox_bytes = (kSlotBytes / 64) * box_rows;                // one value box
      auto load_values = [&](const PUnit& U, int tile, const int64_t* rb, const int* nb) -> bool {
        const int32_t* bt = bt_all + (int64_t)U.b * a.MB;
        for (int kb = 0; kb < 4; ++kb) {
          if (rb[kb] < 0) continue;
          const int valid = U.L - tile * kPairKeys - 64 * kb;
          // a block not loaded whole (boxes past the sequence end) completes its bytes itself
          const bool zero = valid < 64 && ((valid & 15) != 0 || (kSub && nb[kb] < (int)(64 / box_rows)));
          const int tok0 = tile * kPairKeys + 64 * kb;
          const uint32_t slot = r % kRing;
          bool w_ok = lane != 0 || wait(b_empty + 8 * slot, ((r / kRing) & 1) ^ 1);
          if (!__all_sync(0xffffffffu, w_ok)) return false;
          const uint32_t dst = sR + slot * kSlotBytes, lb = lead(b_full + 8 * slot);
          const int32_t c0 = 4 * (int)rank;            // this CTA's value columns 256 rank ..
          if (leader && lane == 0) mbar_arrive_expect_tx(b_full + 8 * slot, 2 * kSlotBytes);
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
            // slot layout [8 key groups][4 chunks][8 rows][128 B]: zero whole rows
            const int nrow = ((valid + 15) & ~15) - valid;
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
              mbar_complete_tx_cluster(lb, kSlotBytes);   // this CTA's share of the slot is in place
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
        // re-reads of long sequences' units
        bool w_ok = lane != 0 || wait(b_qempty, (uq & 1) ^ 1);
        ok = __all_sync(0xffffffffu, w_ok);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t lb = lead(b_qfull);
          if (leader) mbar_arrive_expect_tx(b_qfull, 2 * kPairQBytes);
          if (a.q_whole_rows)       // one box of 64 whole rows: [8 groups][9 chunks][8 rows][128 B]
            tma_load_5d_pair_hint(sQ, &a.tm_q, lb, 0, 0, 0, (128 * U.g + 64 * (int)rank) / 8, U.b, pol_keep);
          else                      // 9 boxes of one 64-column chunk: [9 chunks][64 rows][128 B]
            for (int c = 0; c < 9; ++c)
              tma_load_3d_pair_hint(sQ + c * kQChunk, &a.tm_q, lb, 64 * c, 128 * U.g + 64 * (int)rank, U.b, pol_keep);
        }
        for (int tile = U.tb; tile < U.te && ok; ++tile) {
          int64_t rb[4];
          int nb[4];
          block_rows<kSub>(a, U, tile, rb, nb);
          const int32_t* bt = bt_all + (int64_t)U.b * a.MB;
          // bytes of both CTAs' key halves (the even CTA arms the barrier for both)
          const uint32_t nbox = (uint32_t)(nb[0] + nb[1] + nb[2] + nb[3]);
          for (int ks = 0; ks < kKeySlots; ++ks) {
            const uint32_t slot = r % kRing;
            w_ok = lane != 0 || wait(b_empty + 8 * slot, ((r / kRing) & 1) ^ 1);
            ok = __all_sync(0xffffffffu, w_ok);
            if (!ok) break;
            if (lane == 0) {
              // chunks 2ks, 2ks + 1 (the last slot: chunk 8 and a zero-filled chunk past the row)
              const uint32_t lb = lead(b_full + 8 * slot), dst = sR + slot * kSlotBytes;
              if (leader) mbar_arrive_expect_tx(b_full + 8 * slot, nbox * kbox_bytes);
              for (int h = 0; h < 2; ++h) {
                const int kb = 2 * (int)rank + h;
                if (nb[kb] == 0) continue;
                const uint32_t d = dst + h * (kSlotBytes / 2);
                tma_load_4d_pair_hint(d, &a.tm_k, lb, 0, 0, 2 * ks, (int32_t)(rb[kb] >> 3), pol_keep);
                if (kSub && nb[kb] > 1)
                  load_more_boxes(kBoxPairHint, &a.tm_k, d, lb, 2 * ks, kbox_bytes, bt, a, tile * kPairKeys + 64 * kb,
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
      // after an abort the odd CTA cannot observe its own loads (they count on the even CTA's
      // barrier, whose phase may never complete): both producers wait 50 us, far longer than
      // a load takes, before leaving
      if (*abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 50000ull) {
        }
      }
      // the even CTA waits until the last loads of both CTAs have landed (normally the MMA
      // issuer already has); a CTA must not leave with copies into its memory in flight
      if (leader && lane == 0) {
        volatile uint32_t no_abort = 0;
        for (uint32_t q = r > (uint32_t)kRing ? r - kRing : 0; q < r; ++q)
          mbar_wait(b_full + 8 * (q % kRing), (q / kRing) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
        if (uq > 0) mbar_wait(b_qfull, (uq - 1) & 1, &no_abort, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);
      }
      }
    } else if (warp == 1 && leader) {
      // ================================================================ MMA issuer (even CTA)
      if (lane == 0) {
        // operands bf16, or fp16 for the FP8 cache (E4M3 -> fp16 is exact)
        const uint32_t idesc_qk = make_idesc(256, 128, FP8 ? 0u : 1u, 0, 0);
        const uint32_t idesc_pv = make_idesc(256, 128, FP8 ? 0u : 1u, 1, 1);
        // key slot [2 halves][8 groups][2 chunks][8 rows][128 B]: K-major, 8-row groups 2 KB apart
        const uint64_t dK0 = make_sdesc(sR, 16, 2048, kSwizzle128);
        // Q chunk c: [64 rows][128 B] at sQ + 8 KB c, or chunk c of [8 groups][9 chunks][8 rows]
        const uint64_t dQ0 = make_sdesc(sQ, 16, a.q_whole_rows ? 9 * 1024 : 1024, kSwizzle128);
        const uint32_t q_chunk = a.q_whole_rows ? 1024 : kQChunk;
        // value slot [8 groups][4 chunks][8 rows][128 B]: MN-major, chunks 1 KB, groups 4 KB apart
        const uint64_t dV0 = make_sdesc(sR, 1024, 4096, kSwizzle128);
        const uint64_t dP0 = make_sdesc(sP, 1024, 1024, kSwizzle128);   // MN-major P^T
        uint32_t r = 0, n = 0, uc = 0, pvn = 0, kp = 0;   // kp: FP8 key positions
        bool ok = true;
        struct Prev {
          int L, tile;
          bool first;
          uint32_t uc;
        } prev{0, -1, false, 0};
        auto issue_pv = [&](const Prev& pv) -> bool {
          if (!wait(b_pfull, pvn & 1)) return false;
          if (FP8) fence_proxy_async_smem();   // P^T rows that came by st.async, for the MMAs
          if (pv.first && !wait(b_oempty, (pv.uc & 1) ^ 1)) return false;
          for (int kb = 0; kb < 4; ++kb) {
            const int valid = pv.L - pv.tile * kPairKeys - 64 * kb;
            if (valid <= 0) continue;
            const int ksteps = valid >= 64 ? 4 : (valid + 15) / 16;
            const uint32_t slot = r % kRing;
            if (!wait(b_full + 8 * slot, (r / kRing) & 1)) return false;
            tc_fence_after();
            const uint64_t ad = dV0 + (uint64_t)(slot * (kSlotBytes >> 4));
            const uint64_t bd = dP0 + (uint64_t)((64 * kb * 128) >> 4);
            // M-tile j: output rows 128j.. of each CTA's 256 value columns (its chunks 2j, 2j+1)
            for (int j = 0; j < 2; ++j)
              for (int kk = 0; kk < ksteps; ++kk)
                umma_pair_f16(tmem + kOCol + 128 * j, ad + (uint64_t)((2048 * j + 8192 * kk) >> 4),
                              bd + kk * (2048 >> 4), idesc_pv, !(pv.first && kb == 0 && kk == 0));
            umma_pair_commit(b_empty + 8 * slot);
            ++r;
          }
          umma_pair_commit(b_pvdone);
          ++pvn;
          return true;
        };
        for (int u = u0; u < u1 && ok; ++u, ++uc) {
          const PUnit U = load_punit(a, u);
          ok = wait(FP8 ? b_qready : b_qfull, uc & 1);   // FP8: converted to fp16 in both CTAs
          for (int k = 0; k < U.te - U.tb && ok; ++k, ++n) {
            // S^T buffer: two alternating (bf16), or one (FP8)
            const uint32_t sb = FP8 ? 0u : (n & 1), sph = FP8 ? (n & 1) : ((n >> 1) & 1);
            ok = wait(b_sempty + 8 * sb, sph ^ 1);
            const uint32_t d = tmem + sb * 128;
            for (int ks = 0; ks < kKeySlots && ok; ++ks) {
              const int nc = ks == kKeySlots - 1 ? 1 : 2;     // chunks 2ks, 2ks + 1 (the last: 8)
              if constexpr (FP8) {
                const uint32_t kslot = kp % kKeyTSlots;
                ok = wait(b_kfull + 8 * kslot, (kp / kKeyTSlots) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t at0 = tmem + kKeyCol + 64 * kslot;     // 32 columns per chunk
                for (int cc = 0; cc < nc; ++cc) {
                  const int c = 2 * ks + cc;
                  const uint64_t bd = dQ0 + (uint64_t)(c * (q_chunk >> 4));
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    umma_pair_f16_ts(d, at0 + 32 * cc + 8 * kk, bd + 2 * kk, idesc_qk, (c | kk) != 0);
                }
                umma_pair_commit(b_kempty + 8 * kslot);
                ++kp;
              } else {
                const uint32_t slot = r % kRing;
                ok = wait(b_full + 8 * slot, (r / kRing) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad = dK0 + (uint64_t)(slot * (kSlotBytes >> 4));
                for (int cc = 0; cc < nc; ++cc) {
                  const int c = 2 * ks + cc;
                  const uint64_t bd = dQ0 + (uint64_t)(c * (q_chunk >> 4));
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    umma_pair_f16(d, ad + (uint64_t)(cc * (1024 >> 4) + 2 * kk), bd + 2 * kk, idesc_qk, (c | kk) != 0);
                }
                umma_pair_commit(b_empty + 8 * slot);
                ++r;
              }
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
  }
  } else if (FP8 && warp >= 12) {
    if constexpr (FP8) regs_lower<kRegsConv>();
    // ================================================================ converters (FP8)
    // Warps 12-15 take the raw slots in ring order, with the exact hardware convert (two
    // bytes per instruction). Keys: thread gi converts key row gi of a key position (two
    // chunks) into tensor-memory key slot kp % 2 at lane gi, from which the QK^T MMAs read
    // their A operand (key rows past the sequence end are masked by the softmax). Values:
    // the slot is written as the fp16 operand slot [8 groups][4 chunks][8 rows][128 B]
    // (MN-major, 128-byte swizzled as a TMA load of bf16 rows would land), rows past the
    // sequence end as zeros (the cache may hold NaN there, and 0 * NaN is NaN inside the
    // MMA). Each unit's Q is converted from bf16 to fp16 in place first (a value beyond the
    // fp16 range is flagged). The even CTA's MMA issuer needs both CTAs' halves of a slot:
    // the even CTA's converters arrive on its barrier expecting 16 bytes, which the odd CTA's
    // send with st.async (a remote arrival would hold the sending thread for ~0.85 us).
    const int gi = threadIdx.x - 384;
    constexpr uint32_t cbar = 3;                   // named barrier of the 128 converting threads
    uint32_t rr = 0, fr = 0, kp = 0, uq = 0;       // raw slots, value slots, key positions, units
    bool ok = true;
    auto signal_lead = [&](uint32_t bar) {
      if (leader) mbar_arrive_expect_tx(bar, 16);
      else st_async_v4(lead(smem_u32(sig_s)), make_uint4(0u, 0u, 0u, 0u), lead(bar));
    };
    // key row gi of a raw key slot [2 halves][8 groups][2 chunks][8 rows][64 B], 64-byte
    // swizzled (the 16-byte unit u of row r at u ^ ((r / 2) % 4)), so that the 32 rows a
    // warp reads fall in distinct banks
    const int kr7 = gi & 7;
    const uint32_t krow_off = (uint32_t)(gi >> 6) * (kRawSlotBytes / 2) + (uint32_t)((gi >> 3) & 7) * 1024u +
                              (uint32_t)kr7 * 64u;
    const uint32_t lane_base = tmem + ((uint32_t)(warp & 3) << 21);   // lanes 32 (warp % 4) ..
    auto convert_keys = [&]() -> bool {
      const uint32_t rs = rr % kRawRing, ks = kp % kKeyTSlots;
      const bool mine = gi != 0 || (wait(b_rfull + 8 * rs, (rr / kRawRing) & 1) &&
                                    wait(b_kempty + 8 * ks, ((kp / kKeyTSlots) & 1) ^ 1));
      if (named_bar_or(cbar, 128, !mine)) return false;
      tc_fence_after();
      const uint8_t* src = gRaw + rs * kRawSlotBytes + krow_off;
      const uint32_t tbase = lane_base + kKeyCol + 64 * ks;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint4 raw4[4];
#pragma unroll
        for (int u16 = 0; u16 < 4; ++u16)
          raw4[u16] = *reinterpret_cast<const uint4*>(src + cc * 512 + ((u16 ^ ((kr7 >> 1) & 3)) << 4));
        uint32_t w[32];
#pragma unroll
        for (int u16 = 0; u16 < 4; ++u16) {
          const uint32_t b4[4] = {raw4[u16].x, raw4[u16].y, raw4[u16].z, raw4[u16].w};
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            w[8 * u16 + 2 * k2] = e4m3x2_to_f16x2(b4[k2] & 0xFFFFu);
            w[8 * u16 + 2 * k2 + 1] = e4m3x2_to_f16x2(b4[k2] >> 16);
          }
        }
        tmem_st16u(tbase + 32 * cc, w);
        tmem_st16u(tbase + 32 * cc + 16, w + 16);
      }
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(cbar, 128);
      if (gi == 0) {
        mbar_arrive(b_rempty + 8 * rs);
        signal_lead(b_kfull + 8 * ks);
      }
      ++rr;
      ++kp;
      return true;
    };
    // one 64-key value block: raw slot rr [8 groups][4 chunks][8 rows][64 B] into value slot
    // fr; rows at or past `valid` are zeros
    auto convert_value_slot = [&](int valid) -> bool {
      const uint32_t rs = rr % kRawRing, fs = fr % kRing;
      const bool mine = gi != 0 || (wait(b_rfull + 8 * rs, (rr / kRawRing) & 1) &&
                                    wait(b_empty + 8 * fs, ((fr / kRing) & 1) ^ 1));
      if (named_bar_or(cbar, 128, !mine)) return false;
      const uint8_t* src = gRaw + rs * kRawSlotBytes;
      uint8_t* dst = gR + fs * kSlotBytes;
#pragma unroll 2
      for (int j = 0; j < 8; ++j) {
        // 16-byte raw unit idx: column q4 of row `row` of the 1 KB operand block idx / 32
        // (group idx / 128, chunk (idx / 32) % 4)
        const int idx = gi + 128 * j, q4 = idx & 3, row = (idx >> 2) & 7;
        uint4 v = *reinterpret_cast<const uint4*>(src + 16 * idx);
        if ((idx >> 7) * 8 + row >= valid) v = make_uint4(0u, 0u, 0u, 0u);
        const uint32_t b4[4] = {v.x, v.y, v.z, v.w};
        uint32_t hh[8];
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          hh[2 * k2] = e4m3x2_to_f16x2(b4[k2] & 0xFFFFu);
          hh[2 * k2 + 1] = e4m3x2_to_f16x2(b4[k2] >> 16);
        }
        uint8_t* drow = dst + (idx >> 5) * 1024 + row * 128;
        *reinterpret_cast<uint4*>(drow + (((2 * q4) ^ row) << 4)) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
        *reinterpret_cast<uint4*>(drow + (((2 * q4 + 1) ^ row) << 4)) = make_uint4(hh[4], hh[5], hh[6], hh[7]);
      }
      fence_proxy_async_smem();
      named_bar_sync(cbar, 128);
      if (gi == 0) {
        mbar_arrive(b_rempty + 8 * rs);
        signal_lead(b_full + 8 * fs);
      }
      ++rr;
      ++fr;
      return true;
    };
    auto convert_values = [&](const PUnit& U, int tile) -> bool {
      for (int kb = 0; kb < 4; ++kb) {
        const int valid = U.L - tile * kPairKeys - 64 * kb;
        if (valid > 0 && !convert_value_slot(valid)) return false;
      }
      return true;
    };
    for (int u = u0; u < u1 && ok; ++u, ++uq) {
      const PUnit U = load_punit(a, u);
      // ---- Q, bf16 -> fp16 in place (the 128-byte swizzle moves whole 16-byte units)
      {
        const bool mine = gi != 0 || wait(b_qraw, uq & 1);
        if (named_bar_or(cbar, 128, !mine)) { ok = false; break; }
        bool q_bad = false;
        for (int i = gi; i < kPairQBytes / 16; i += 128) {
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
        named_bar_sync(cbar, 128);
        if (gi == 0) signal_lead(b_qready);
      }
      int pt = -1;
      for (int tile = U.tb; tile < U.te && ok; ++tile) {
        for (int ks = 0; ks < kKeySlots && ok; ++ks) ok = convert_keys();
        if (ok && pt >= 0) ok = convert_values(U, pt);
        pt = tile;
      }
      if (ok && pt >= 0) ok = convert_values(U, pt);
    }
  } else if (warp >= 4) {
    if constexpr (FP8) regs_raise<kRegsSoftmax>();
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
        const uint32_t sb = FP8 ? 0u : (n & 1), sph = FP8 ? (n & 1) : ((n >> 1) & 1);   // S^T buffer
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
        if ((tile + 1) * kPairKeys <= mask_from) {
#pragma unroll
          for (int r = 0; r < 64; r += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mref + r);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              s[r + i] *= c_log2;
              need |= s[r + i] > mm[i] + kPairRescaleLog2;
            }
          }
        } else {
#pragma unroll
          for (int r = 0; r < 64; r += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mref + r);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              s[r + i] = j < nvis_s[wg][r + i] ? s[r + i] * c_log2 : -INFINITY;
              need |= s[r + i] > mm[i] + kPairRescaleLog2;
            }
          }
        }
        // the barrier also orders every thread's S^T reads before the even CTA's signal
        const bool need_local = named_bar_or(bar, 128, need);
        // bf16: the odd CTA's S^T reads precede its P^T signal, which the MMA issuer awaits
        // before it reuses the buffer two tiles later. FP8 (one S^T buffer): the even CTA's
        // warpgroups arrive expecting 16 bytes each, which the odd CTA's warpgroups send by
        // st.async once their reads are done.
        if (t == 0) {
          if (!FP8) {
            if (leader) mbar_arrive(b_sempty + 8 * sb);
          } else if (leader) {
            mbar_arrive_expect_tx(b_sempty + 8 * sb, 16);
          } else {
            st_async_v4(lead(smem_u32(sig_s)), make_uint4(0u, 0u, 0u, 0u), lead(b_sempty + 8 * sb));
          }
        }
        if (need_local) {
          // column maxima of the warp's 32 keys for all 64 rows at once (reduce-scatter,
          // as for the row sums; shuffles rather than 64 redux operations, which the
          // converting warps' convert instructions slow down in the FP8 kernel)
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
        uint32_t pw[32];
#pragma unroll
        for (int r = 0; r < 64; r += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(mref + r);
          const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int i = 0; i < 4; i += 2) {
            const float p0 = s[r + i] == -INFINITY ? 0.f : ex2_approx(s[r + i] - mm[i]);
            const float p1 = s[r + i + 1] == -INFINITY ? 0.f : ex2_approx(s[r + i + 1] - mm[i + 1]);
            if constexpr (FP8) {                 // the MMA operand type: fp16 with the FP8 cache
              __half2 h = __floats2half2_rn(p0, p1);
              pw[(r + i) / 2] = *reinterpret_cast<uint32_t*>(&h);
            } else {
              __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
              pw[(r + i) / 2] = *reinterpret_cast<uint32_t*>(&h);
            }
            lsum[r + i] += p0;                 // the normaliser sums the unrounded values
            lsum[r + i + 1] += p1;
          }
        }
        // P^T and O^T are free once the previous PV has completed; the staging buffer once
        // the previous copy out of it has been read
        if (!FP8 && t == 0 && !local_p) bulk_wait_read0();
        // FP8: the other warpgroup's previous epilogue used the upper half of this P^T region
        if (FP8 && local_p && k == 0 && ui > 0) {
          ok = wait_wg(b_epi, (ui - 1) & 1);
          if (!ok) break;
        }
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
        // the peer, into the staging buffer laid out as the peer's P^T rows 128 rank ..
        // 128 rank + 127 (bf16), or straight into the peer's P^T by st.async, its bytes
        // counted on the peer's barrier (FP8: no room for a staging buffer)
        if (FP8 && !local_p) {
          const uint32_t pdst = map_to_rank(sP + (uint32_t)rank * kStageBytes, peer);
          const uint32_t pbar = map_to_rank(leader ? b_pin : b_pfull, peer);
#pragma unroll
          for (int u16 = 0; u16 < 8; ++u16)
            st_async_v4(pdst + p_off128(t, u16), make_uint4(pw[4 * u16], pw[4 * u16 + 1], pw[4 * u16 + 2], pw[4 * u16 + 3]),
                        pbar);
        } else {
          uint8_t* prow = local_p ? gP + 128 * (int)rank * 128 : gStage;
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
            // rows for the peer's P^T: one bulk copy, counted on the peer's barrier (the even
            // CTA's P^T barrier, or the odd CTA's b_pin); FP8: already sent
            if (!FP8) {
              bulk_copy_to_cluster(map_to_rank(sP + (uint32_t)rank * kStageBytes, peer), sStage, kStageBytes,
                                   map_to_rank(leader ? b_pin : b_pfull, peer));
              bulk_commit();
            }
          } else if (leader) {
            mbar_arrive_expect_tx(b_pfull, kStageBytes);   // own rows; the odd CTA's copy to come
          } else {
            mbar_arrive_expect_tx(b_pin, kStageBytes);
            ok = mbar_wait(b_pin, n & 1, abort_flag, err, MLA_DEVERR_TIMEOUT, a.wait_limit_ns);   // the even CTA's copy
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
      // rows per load. It transposes them through 2 KB of shared memory, 16-byte blocks
      // XOR-swizzled by row, so that each lane stores 16 consecutive columns of one row
      // (16-byte stores instead of one store per row and column). The scratch is this CTA's
      // own half of the P^T buffer for the warpgroup whose rows live here (no other agent
      // writes it before this warpgroup's next P^T), else the staging buffer once its last
      // copy to the peer has been read.
      // FP8 has no staging buffer: its other warpgroup uses the upper half of the same
      // region, and the P^T rows of the next unit wait for it (b_epi).
      if (!FP8 && !local_p) {
        if (t == 0) bulk_wait_read0();
        named_bar_sync(bar, 128);
      }
      uint8_t* scratch = local_p ? gP + (int)rank * kStageBytes : FP8 ? gP + (int)rank * kStageBytes + 8192 : gStage;
      float* stage = reinterpret_cast<float*>(scratch) + wl * 512;
      const int nrows = min(64, R - row0);         // rows of this warpgroup that exist
      const int si = lane >> 1, sh = lane & 1;
#pragma unroll 1
      for (int jt = 0; jt < 2; ++jt) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float o[16];
          tmem_ld16(tmem + lane_addr + kOCol + 128 * jt + 64 * wg + 16 * c, o);
          tmem_wait_ld();
          if (jt == 1 && c == 3) {
            // O^T has been read: the next unit's first PV may overwrite it
            tc_fence_before();
            named_bar_sync(bar, 128);
            if (leader && t == 0) mbar_arrive(b_oempty);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            stage[i * 32 + ((((lane >> 2) ^ (i & 7)) << 2) | (lane & 3))] = o[i] * alpha_s[wg][16 * c + i];
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
          const int r = 16 * c + si;               // row 64 wg + r of the unit
          const int col = 256 * (int)rank + 128 * jt + 32 * wl + 16 * sh;
          if (r < nrows) {
            if (direct) {
              uint32_t w[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
                w[k] = *reinterpret_cast<uint32_t*>(&h);
              }
              uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)U.b * R + row0 + r) * kDV + col);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
              float4* dst = reinterpret_cast<float4*>(a.part_o + ((int64_t)U.slot * 128 + 64 * wg + r) * kDV + col);
#pragma unroll
              for (int m = 0; m < 4; ++m) dst[m] = make_float4(v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]);
            }
          }
        }
      }
      if (rank == 0 && t < 64 && row0 + t < R) {
        const float l = tot > 0.f ? (mref[t] + __log2f(tot)) * kPLn2 : -INFINITY;
        if (direct) a.lse[(int64_t)U.b * R + row0 + t] = l;
        else a.part_lse[(int64_t)U.slot * 128 + 64 * wg + t] = l;
      }
      named_bar_sync(bar, 128);
      if (FP8 && !local_p && t == 0) mbar_arrive(b_epi);   // its scratch reads are done
      gn += T;
    }
    // a copy out of the staging buffer has landed before the CTA may leave
    if (t == 0 && !local_p) bulk_wait0();
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
  using Cfg = PairCfg<FP8>;
  cudaError_t e = cudaFuncSetAttribute(decode_pair_kernel<FP8, kSub>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kDynBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, decode_pair_kernel<FP8, kSub>);
  if (e != cudaSuccess) return e;
  if ((int)attr.sharedSizeBytes > kPairStaticBudget) return cudaErrorInvalidConfiguration;
  // the FP8 kernel's register budgets redistribute exactly 128 registers per thread
  if (FP8 && attr.numRegs != 128) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

template <bool FP8>
static cudaError_t launch_pair_variant(const DecodeArgs& a, int pairs, cudaStream_t s) {
  using Cfg = PairCfg<FP8>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kDynBytes;
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
