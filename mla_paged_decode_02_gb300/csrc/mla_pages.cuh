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
#include "../../include/mla.h"

namespace mla {

// Cache row of token `tok` of the sequence whose block-table row is `bt`. An entry outside
// the pool is reported in the error word (when `report`) and page 0 is read instead.
__device__ __forceinline__ int64_t page_row(const int32_t* bt, int tok, const DecodeArgs& a, uint32_t* err,
                                            bool report) {
  const int pg = __ldg(bt + tok / a.P);
  if (pg < 0 || pg >= a.num_pages) {
    if (report) atomicOr(err, MLA_DEVERR_BLOCK_TABLE);
    return tok % a.P;
  }
  return (int64_t)pg * a.P + tok % a.P;
}

// Boxes of the block with `valid` rows before the sequence end (<= 0: none) that are loaded.
__device__ __forceinline__ int block_boxes(int valid, int box_rows) {
  if (valid <= 0) return 0;
  const int n = (valid + box_rows - 1) / box_rows, per = 64 / box_rows;
  return n < per ? n : per;
}

// Issues the `nbox` boxes of the block starting at token `tok0` whose first box starts at
// cache row `row0`: issue(k, first 8-row group of box k). Boxes after the first look their
// page up again (and report a bad entry).
template <class F>
__device__ __forceinline__ void issue_block(const int32_t* bt, const DecodeArgs& a, uint32_t* err, int tok0,
                                            int64_t row0, int nbox, F&& issue) {
  issue(0, (int32_t)(row0 >> 3));
  for (int k = 1; k < nbox; ++k) issue(k, (int32_t)(page_row(bt, tok0 + k * a.box_rows, a, err, true) >> 3));
}

}  // namespace mla
