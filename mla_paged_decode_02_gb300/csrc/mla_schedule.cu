// mla_schedule.cu — on-device split-KV scheduler (one CTA).
//
// "[NVIDIA] Add Cutlass MLA backend" (review thread) shows FlashAttention's
// ahead-of-time scheduler, get_scheduler_metadata(batch_size, max_seqlen_k,
// cache_seqlens, num_heads, headdim, page_size, causal, ...), which turns the
// per-sequence lengths into a work partition before the attention kernel runs. This is
// our own version of that step, computed on the device from seq_lens so that the whole
// decode stays free of host synchronisation.
//
// Work is counted in (key tile, row group) pairs. Sequence b has n_b = ceil(L_b / T)
// key tiles (T = 128, or 256 for CTA pairs) and G groups of query rows; each (g, b) is a
// stream of X + n_b positions — X for the set-up of a unit (loading and converting its
// q, refilling the pipeline, its epilogue; about two tiles of streaming) and one per tile —
// and the streams are laid end to end, group-major:
//   pos(g, b) = g * N + sum_{b' < b} (X + n_b'),    N = sum_b (X + n_b),    W = G * N,
// The persistent decode grid has one CTA per SM; CTA c takes the positions
// [c q, (c + 1) q) with q = ceil(W / grid), i.e. the tiles among them, so no CTA has
// more than one tile more work than another (counting a unit's set-up) whatever the length
// mix. X is dropped when a CTA's share would be too small for it (q <= 2 X): then every
// CTA range holds at least one tile. When G divides the grid, each row group instead
// gets exactly grid / G CTAs and the same partition of its N tiles (q = ceil(N G / grid)):
// CTA c + k grid / G then reads the same key tiles as CTA c, in the same order and at about
// the same time, so of the G reads of every key tile only the first comes from DRAM. A stream that a CTA boundary cuts becomes one
// unit per CTA it touches; each such piece writes a partial output (normalised, with
// its log-sum-exp) to its own slot, and the combine kernel merges the pieces. Streams
// inside one CTA write the final output directly. Units are stored in position order,
// so the units of CTA c are the contiguous range [cta_first[c], cta_first[c + 1]).
// The G x B streams are handled as one flattened, position-ordered index space (each
// thread a contiguous range of it, one block-wide scan for the unit, split and slot
// offsets), so the schedule's cost does not grow with the number of row groups.
#include "mla_cache_write.cuh"
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "../../include/mla.h"

namespace mla {

constexpr int kSchedThreads = 1024;
constexpr int kMaxWriteCtas = 128;
constexpr int kMaxGroups = kMaxRows / 16;   // row groups of a sequence (16 rows or more each)

// Exclusive prefix sum over the block's threads (warp shuffles, then the 32 warp totals).
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* tmp, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = tmp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    tmp[lane] = w;                         // inclusive totals of warps 0..lane
  }
  __syncthreads();
  const int64_t before = (warp > 0 ? tmp[warp - 1] : 0) + x - v;
  *total = tmp[31];
  __syncthreads();
  return before;
}

__device__ __forceinline__ int clamped_len(const SchedArgs& a, int b, bool report) {
  const int L = a.seq_lens[b];
  const int Lc = L < a.s_q ? a.s_q : (L > a.max_len ? a.max_len : L);
  if (report && Lc != L) atomicOr(a.hdr, MLA_DEVERR_SEQ_LEN);
  return Lc;
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(SchedArgs a) {
  static_assert(kSchedThreads == 1024, "the scan assumes 32 warps");
  __shared__ int64_t scan_tmp[32];
  __shared__ int64_t n_tiles_s;
  __shared__ int32_t gend_s[kMaxGroups];   // end of each row group's units (aligned mode)
  const int tid = threadIdx.x;
  griddep_launch_dependents();         // the decode grid may start its set-up now
  if (blockIdx.x > 0) {
    // fused call: CTAs 1.. write the step's new tokens into the cache while CTA 0 computes
    // the schedule (the decode grid reads the cache only after this grid has completed).
    // Slots outside the pool are skipped here and reported by the combine kernel, which
    // runs after CTA 0 has cleared the error word.
    const int64_t total = (int64_t)a.w_n * kWriteGroupsPerToken;
    const int64_t stride = (int64_t)(gridDim.x - 1) * kSchedThreads;
    const float scale = a.w_fp8 ? __ldg(a.w_kv_scale) : 1.0f;
    for (int64_t i = (int64_t)(blockIdx.x - 1) * kSchedThreads + tid; i < total; i += stride) {
      const int64_t t = i / kWriteGroupsPerToken;
      const int c = (int)(i - t * kWriteGroupsPerToken);
      if (a.w_fp8) write_group<true>(a.w_latent, a.w_rope, a.w_slots, t, c, a.w_cache, a.w_total_slots, scale, nullptr);
      else write_group<false>(a.w_latent, a.w_rope, a.w_slots, t, c, a.w_cache, a.w_total_slots, scale, nullptr);
    }
    return;
  }
  if (tid == 0) a.hdr[0] = 0u;
  __syncthreads();

  const int G = a.G, B = a.B;
  // 1. key tiles per sequence (lengths clamped into the valid range; bad ones flagged) and
  //    their exclusive prefix: batch_info[b] = (tiles, first tile of b, clamped length, 0)
  {
    const int chunk = (B + kSchedThreads - 1) / kSchedThreads;
    const int b0 = tid * chunk, b1 = min(B, b0 + chunk);
    int64_t my_tiles = 0;
    for (int b = b0; b < b1; ++b) my_tiles += (clamped_len(a, b, true) + a.tile - 1) / a.tile;
    int64_t n_tiles_all;
    int64_t off = block_exclusive_scan(my_tiles, scan_tmp, &n_tiles_all);
    for (int b = b0; b < b1; ++b) {
      const int Lc = clamped_len(a, b, false);
      const int n = (Lc + a.tile - 1) / a.tile;
      a.batch_info[b] = make_int4(n, (int)off, Lc, 0);
      off += n;
    }
    if (tid == 0) n_tiles_s = n_tiles_all;
  }
  __syncthreads();                     // batch_info (global, this block's writes) and n_tiles_s
  const int64_t n_tiles = n_tiles_s;
  const bool aligned = G > 1 && a.grid % G == 0;   // one CTA block per row group
  const int cpg = aligned ? a.grid / G : a.grid;    // CTAs per row group
  int X = a.setup > 0 ? a.setup : 0;
  int64_t Nv = n_tiles + (int64_t)B * X;            // positions of one row group
  int64_t q = aligned ? (Nv + cpg - 1) / cpg : ((int64_t)G * Nv + a.grid - 1) / a.grid;   // >= 1
  if (X > 0 && q <= 2 * (int64_t)X) {
    X = 0;
    Nv = n_tiles;
    q = aligned ? (Nv + cpg - 1) / cpg : ((int64_t)G * Nv + a.grid - 1) / a.grid;
  }

  // 2. the (row group g, sequence b) streams in position order, flattened: item i = g B + b,
  //    stream start pos = (aligned ? 0 : g N) + b X + first tile of b, its tiles from
  //    pos + X on. Every stream is cut at the CTA boundaries its tiles cross (multiples of
  //    q): ns pieces, one unit each; a cut stream (ns >= 2) gets ns consecutive partial
  //    slots and an entry in the split list.
  const int64_t items = (int64_t)G * B;
  const int64_t ichunk = (items + kSchedThreads - 1) / kSchedThreads;
  const int64_t i0 = (int64_t)tid * ichunk, i1 = min(items, i0 + ichunk);
  auto pieces = [&](int64_t i, int64_t* pre_out, int* n_out) -> int64_t {
    const int g = (int)(i / B), b = (int)(i - (int64_t)g * B);
    const int4 bi = a.batch_info[b];
    const int64_t pre = (aligned ? 0 : (int64_t)g * Nv) + (int64_t)b * X + bi.y;   // the stream's start
    const int64_t ts = pre + X;                                                        // its first tile
    *pre_out = pre;
    *n_out = bi.x;
    return (ts + bi.x - 1) / q - ts / q + 1;
  };
  int64_t my_units = 0, my_split = 0, my_slots = 0;
  for (int64_t i = i0; i < i1; ++i) {
    int64_t pre;
    int n;
    const int64_t ns = pieces(i, &pre, &n);
    my_units += ns;
    if (ns >= 2) { my_split += 1; my_slots += ns; }
  }
  int64_t n_units, n_split, n_slots;
  int64_t unit_off = block_exclusive_scan(my_units, scan_tmp, &n_units);
  int64_t split_off = block_exclusive_scan(my_split, scan_tmp, &n_split);
  int64_t slot_off = block_exclusive_scan(my_slots, scan_tmp, &n_slots);
  if (n_units > a.max_units || n_split > a.max_split || n_slots > a.max_slots) {
    // cannot happen for the sizes mla_decode_workspace_size returns; refuse to overflow
    for (int c = tid; c <= a.grid; c += kSchedThreads) a.cta_first[c] = 0;
    if (tid == 0) { atomicOr(a.hdr, MLA_DEVERR_SEQ_LEN); a.hdr[1] = 0; a.hdr[2] = 0; }
    return;
  }
  // the first unit of each CTA is set below; a CTA whose range starts at or past the end
  // has no work (patched in step 3)
  for (int c = tid; c <= a.grid; c += kSchedThreads) a.cta_first[c] = -1;
  __syncthreads();
  for (int64_t i = i0; i < i1; ++i) {
    int64_t pre;
    int n;
    const int ns = (int)pieces(i, &pre, &n);
    const int g = (int)(i / B), b = (int)(i - (int64_t)g * B);
    const int cbase = aligned ? g * cpg : 0;
    if (b == 0 && g > 0) gend_s[g - 1] = (int32_t)unit_off;   // the units of groups < g end here
    const int64_t ts = pre + X;
    const int64_t c_lo = ts / q;
    const int slot0 = ns >= 2 ? (int)slot_off : -1;
    if (ns >= 2) a.split_list[split_off++] = make_int4(b, g, ns, slot0);
    for (int k = 0; k < ns; ++k) {
      const int64_t c = c_lo + k;
      const int64_t s0 = ts > c * q ? ts : c * q;
      const int64_t s1 = ts + n < (c + 1) * q ? ts + n : (c + 1) * q;
      const int tb = (int)(s0 - ts), te = (int)(s1 - ts);
      a.units[unit_off] = make_int4(b, g, tb | (te << 16), ns >= 2 ? slot0 + k : -1);
      // the CTA's first unit: its range starts at this piece, or inside this stream's set-up
      if (s0 == c * q || (k == 0 && pre <= c * q)) a.cta_first[cbase + c] = (int32_t)unit_off;
      ++unit_off;
    }
    if (ns >= 2) slot_off += ns;
  }
  if (tid == 0) gend_s[G - 1] = (int32_t)n_units;
  __syncthreads();
  // 3. CTAs without work start (and end) at the end of their group's units (aligned: so
  //    that the ranges [cta_first[c], cta_first[c + 1]) stay within the group), else at
  //    the end of all units
  for (int c = tid; c <= a.grid; c += kSchedThreads)
    if (a.cta_first[c] < 0) a.cta_first[c] = aligned && c < a.grid ? gend_s[c / cpg] : (int32_t)n_units;
  if (tid == 0) {
    a.hdr[1] = (uint32_t)n_units;
    a.hdr[2] = (uint32_t)n_split;
    a.hdr[3] = (uint32_t)(q < 0xFFFFFFFFll ? q : 0xFFFFFFFFll);
    a.hdr[4] = (uint32_t)X;
  }
}

cudaError_t launch_schedule(const SchedArgs& a, cudaStream_t s) {
  // CTA 0 schedules; a fused cache write adds CTAs of 1024 threads, one 8-value group each
  int extra = 0;
  if (a.w_n > 0) {
    const int64_t groups = (int64_t)a.w_n * kWriteGroupsPerToken;
    extra = (int)((groups + kSchedThreads - 1) / kSchedThreads);
    if (extra > kMaxWriteCtas) extra = kMaxWriteCtas;
  }
  schedule_kernel<<<1 + extra, kSchedThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
