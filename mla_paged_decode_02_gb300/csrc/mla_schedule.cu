// mla_schedule.cu — on-device split-KV scheduler (one CTA).
//
// "[NVIDIA] Add Cutlass MLA backend" (review thread) shows FlashAttention's
// ahead-of-time scheduler, get_scheduler_metadata(batch_size, max_seqlen_k,
// cache_seqlens, num_heads, headdim, page_size, causal, ...), which turns the
// per-sequence lengths into a work partition before the attention kernel runs. This is
// our own version of that step, computed on the device from seq_lens so that the whole
// decode stays free of host synchronisation:
//
//   n_b  = ceil(L_b / 128)                      key tiles of sequence b
//   C    = max(1, ceil(G * sum_b n_b / target)) tiles per split, target = 2 * #SMs
//   ns_b = ceil(n_b / C)                        splits of sequence b; split s covers
//          tiles [floor(s n_b / ns_b), floor((s+1) n_b / ns_b))
//
// Every split becomes G units (one per group of query rows). Units are emitted
// longest-first (a counting sort on the tile count) so that the persistent decode grid,
// which walks them with a static stride, finishes evenly. Sequences with ns_b >= 2
// get partial-output slots for the LSE combine; the others write the final output.
#include "mla_internal.h"
#include "../../include/mla.h"

namespace mla {

constexpr int kSchedThreads = 1024;
constexpr int kMaxTilesPerSeq = kMaxSeqLen / kTileTokens;   // 8192

__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* tmp, int64_t* total) {
  const int tid = threadIdx.x;
  tmp[tid] = v;
  __syncthreads();
  for (int off = 1; off < kSchedThreads; off <<= 1) {
    int64_t add = tid >= off ? tmp[tid - off] : 0;
    __syncthreads();
    tmp[tid] += add;
    __syncthreads();
  }
  const int64_t incl = tmp[tid];
  *total = tmp[kSchedThreads - 1];
  __syncthreads();
  return incl - v;
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(SchedArgs a) {
  __shared__ int64_t scan_tmp[kSchedThreads];
  __shared__ int32_t hist[kMaxTilesPerSeq + 1];
  const int tid = threadIdx.x;
  if (tid == 0) a.hdr[0] = 0u;
  for (int i = tid; i <= kMaxTilesPerSeq; i += kSchedThreads) hist[i] = 0;
  __syncthreads();

  const int chunk = (a.B + kSchedThreads - 1) / kSchedThreads;
  const int b0 = tid * chunk;
  const int b1 = min(a.B, b0 + chunk);
  const int max_len = a.max_len;

  // 1. tiles per sequence (lengths clamped into the valid range; bad ones flagged)
  int64_t my_tiles = 0;
  for (int b = b0; b < b1; ++b) {
    int L = a.seq_lens[b];
    int Lc = L < a.s_q ? a.s_q : (L > max_len ? max_len : L);
    if (Lc != L) atomicOr(a.hdr, MLA_DEVERR_SEQ_LEN);
    my_tiles += (Lc + kTileTokens - 1) / kTileTokens;
  }
  int64_t sum_tiles;
  block_exclusive_scan(my_tiles, scan_tmp, &sum_tiles);
  int64_t C = (a.G * sum_tiles + a.target_units - 1) / a.target_units;
  if (C < 1) C = 1;

  // 2. splits, partial slots and split batches per thread, then block scans
  int64_t my_items = 0, my_pslots = 0, my_splitb = 0;
  for (int b = b0; b < b1; ++b) {
    int L = a.seq_lens[b];
    int Lc = L < a.s_q ? a.s_q : (L > max_len ? max_len : L);
    int n = (Lc + kTileTokens - 1) / kTileTokens;
    int ns = (int)((n + C - 1) / C);
    my_items += ns;
    if (ns >= 2) { my_pslots += ns; my_splitb += 1; }
  }
  int64_t n_items, n_pslots, n_splitb;
  int64_t item_off = block_exclusive_scan(my_items, scan_tmp, &n_items);
  int64_t pslot_off = block_exclusive_scan(my_pslots, scan_tmp, &n_pslots);
  int64_t splitb_off = block_exclusive_scan(my_splitb, scan_tmp, &n_splitb);
  const bool fits = n_items <= a.max_items && n_pslots <= a.max_pslots;
  if (!fits) {
    // cannot happen for the sizes mla_decode_workspace_size returns; refuse to overflow
    if (tid == 0) { atomicOr(a.hdr, MLA_DEVERR_SEQ_LEN); a.hdr[1] = 0; a.hdr[2] = 0; }
    return;
  }

  // 3. per-batch info, split list, unsorted items, size histogram
  for (int b = b0; b < b1; ++b) {
    int L = a.seq_lens[b];
    int Lc = L < a.s_q ? a.s_q : (L > max_len ? max_len : L);
    int n = (Lc + kTileTokens - 1) / kTileTokens;
    int ns = (int)((n + C - 1) / C);
    int pbase = ns >= 2 ? (int)pslot_off : -1;
    a.batch_info[b] = make_int4(ns, pbase, Lc, (int)item_off);
    if (ns >= 2) a.split_list[splitb_off++] = b;
    for (int s = 0; s < ns; ++s) {
      int tb = (int)((int64_t)s * n / ns);
      int te = (int)((int64_t)(s + 1) * n / ns);
      a.items_tmp[item_off + s] = make_int4(b, s, tb | (te << 16), ns >= 2 ? pbase + s : -1);
      atomicAdd(&hist[te - tb], 1);
    }
    item_off += ns;
    if (ns >= 2) pslot_off += ns;
  }
  __syncthreads();

  // 4. start offset of each size class, largest sizes first
  {
    constexpr int kPer = (kMaxTilesPerSeq + 1 + kSchedThreads - 1) / kSchedThreads;   // 9
    // thread tid owns sizes [hi_size - kPer*(tid+1) + 1, hi_size - kPer*tid] in descending order
    int64_t local = 0;
    int sz[kPer];
    for (int k = 0; k < kPer; ++k) {
      int s = kMaxTilesPerSeq - (tid * kPer + k);
      sz[k] = s;
      local += s >= 1 ? hist[s] : 0;
    }
    int64_t tot;
    int64_t run = block_exclusive_scan(local, scan_tmp, &tot);
    for (int k = 0; k < kPer; ++k) {
      int s = sz[k];
      if (s >= 1) {
        int h = hist[s];
        hist[s] = (int)run;
        run += h;
      }
    }
  }
  __syncthreads();

  // 5. scatter items into sorted order; each expands into G consecutive units
  for (int64_t it = tid; it < n_items; it += kSchedThreads) {
    int4 v = a.items_tmp[it];
    int tb = v.z & 0xFFFF, te = (int)((unsigned)v.z >> 16);
    int pos = atomicAdd(&hist[te - tb], 1);
    for (int g = 0; g < a.G; ++g)
      a.units[(int64_t)pos * a.G + g] = make_int4(v.x, g, v.z, v.w);
  }
  if (tid == 0) {
    a.hdr[1] = (uint32_t)(n_items * a.G);
    a.hdr[2] = (uint32_t)n_splitb;
    a.hdr[3] = (uint32_t)C;
  }
}

cudaError_t launch_schedule(const SchedArgs& a, cudaStream_t s) {
  schedule_kernel<<<1, kSchedThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
