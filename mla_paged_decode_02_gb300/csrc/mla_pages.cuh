// mla_pages.cuh — paged-cache addressing shared by the decode kernels.
//
// The cache is [num_pages][P][576]; token j of sequence b is row j % P of page
// block_table[b][j / P] ("[NVIDIA] Add Cutlass MLA backend", review thread: the block
// table maps a sequence's logical blocks to physical pages of page_size tokens).
//
// The kernels fetch keys and values per 64-token block of a key tile. A block is loaded as
// 64 / box_rows TMA boxes of box_rows = gcd(P, 64) rows (P a multiple of 8), so that no box
// straddles two pages: with P a multiple of 64 that is one box per block, with P = 16 four
// boxes from four pages. Box k of a block lands box_rows rows after box k - 1 (the tensor
// maps count rows in 8-row groups, the outermost dimension of a box in shared memory).
// Only boxes that start before the sequence end are loaded; the rows of a box past the end
// are masked (keys) or zeroed (values) by the kernels.
#pragma once
#include <cstdint>
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "../../include/mla.h"

namespace mla {

// Cache row of token `tok` of the sequence whose block-table row is `bt`. An entry outside
// the pool reads page 0 instead (the combine kernel reports it in the error word).
__device__ __forceinline__ int64_t page_row(const int32_t* bt, int tok, const DecodeArgs& a) {
  const int pg = __ldg(bt + tok / a.P);
  if (pg < 0 || pg >= a.num_pages) return tok % a.P;
  return (int64_t)pg * a.P + tok % a.P;
}

// Boxes of the block with `valid` rows before the sequence end (<= 0: none) that are loaded.
// box_rows is a power of two (a divisor of 64).
__device__ __forceinline__ int block_boxes(int valid, int box_rows) {
  if (valid <= 0) return 0;
  const int sh = 31 - __clz(box_rows);
  const int n = (valid + box_rows - 1) >> sh, per = 64 >> sh;
  return n < per ? n : per;
}

enum BoxLoad { kBoxPlain = 0, kBoxHint = 1, kBoxPairHint = 2 };

// Boxes 1 .. nb - 1 of the block starting at token tok0 (pages smaller than 64 rows), each
// looking its page up. Box k lands at dst + k * box_bytes, with
// the mbarrier and the TMA form of box 0. Kept out of line, so that the usual case (one box
// per block) stays small in the instruction cache that a CTA's roles share.
static __device__ __noinline__ void load_more_boxes(int form, const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                             int32_t chunk, uint32_t box_bytes, const int32_t* bt,
                                             const DecodeArgs& a, int tok0, int nb, uint64_t pol) {
  for (int k = 1; k < nb; ++k) {
    const int32_t grp = (int32_t)(page_row(bt, tok0 + k * a.box_rows, a) >> 3);
    const uint32_t d = dst + (uint32_t)k * box_bytes;
    if (form == kBoxPairHint) tma_load_4d_pair_hint(d, map, bar, 0, 0, chunk, grp, pol);
    else if (form == kBoxHint) tma_load_4d_hint(d, map, bar, 0, 0, chunk, grp, pol);
    else tma_load_4d(d, map, bar, 0, 0, chunk, grp);
  }
}

}  // namespace mla
