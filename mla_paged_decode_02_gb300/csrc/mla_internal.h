// mla_internal.h — workspace layout and kernel argument blocks shared by the host API
// (mla_api.cu) and the kernels. Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace mla {

constexpr int kDQK = 576;          // 512 latent + 64 rope
constexpr int kDV = 512;
constexpr int kTileTokens = 128;   // keys per tile: the M of the QK^T MMA (tokens on M)
constexpr int kMaxSeqLen = 1 << 20;
constexpr int kMaxRows = 65536;    // s_q * H
constexpr int kMaxSq = 512;        // new query tokens per sequence (the decode threshold the
                                   // "[WIP][Attention] FlashAttn MLA" page tunes up to)
constexpr int kMaxBatch = 1 << 16;
constexpr int kMaxFusedWriteTokens = 1 << 17;   // new tokens the scheduler's launch writes itself

// Execution plan for the s_q * H query rows of a sequence. Rows are processed in groups
// of RC rows (the N of every MMA). Up to 64 rows: one CTA per SM, RC = 16/32/64, 128-key
// tiles. More than 64 rows: CTA pairs (a cluster of two CTAs on two SMs) with RC = 128
// and 256-key tiles, each CTA holding 128 of the keys and 64 of the rows, so that every
// key tile is read (and, with the FP8 cache, converted) once for 128 rows. The schedule's
// workers are SMs or CTA pairs. The plan is the same for both cache types.
struct Plan {
  int rc, G, tile;
  bool pair;
};
inline Plan make_plan(int rows, bool /*fp8*/) {
  Plan p;
  p.pair = rows > 64;
  p.rc = p.pair ? 128 : rows <= 16 ? 16 : rows <= 32 ? 32 : 64;
  p.G = (rows + p.rc - 1) / p.rc;
  p.tile = p.pair ? 2 * kTileTokens : kTileTokens;
  return p;
}
inline int plan_workers(const Plan& p, int num_sms) { return p.pair ? num_sms / 2 : num_sms; }

// Workspace: [header 256 B][batch_info int4 x B][cta_first int32 x (grid + 1)]
//            [split_list int4 x max_split][units int4 x max_units]
//            [part_lse f32 x max_slots*RC][part_o f32 x max_slots*RC*512]
// header word 0: device error bits; 1: number of units; 2: number of split streams;
// 3: positions per CTA (q); 4: positions charged at the start of every stream (X). The bounds follow from the partition (mla_schedule.cu): every
// CTA boundary cuts at most one (sequence, row group) stream, so there are at most
// B*G + grid - 1 units, grid - 1 split streams and 2*(grid - 1) partial slots.
struct WsLayout {
  size_t batch_off, cta_off, split_off, units_off, plse_off, po_off, total;
  int64_t max_units, max_split, max_slots;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int B, const Plan& p, int grid) {
  WsLayout w{};
  const int rc = p.rc;
  const int64_t G = p.G;
  w.max_units = (int64_t)B * G + grid;
  w.max_split = grid;
  w.max_slots = 2 * (int64_t)grid;
  size_t off = 256;
  w.batch_off = off;  off = align_up(off + sizeof(int4) * (size_t)B, 256);
  w.cta_off = off;    off = align_up(off + sizeof(int32_t) * (size_t)(grid + 1), 256);
  w.split_off = off;  off = align_up(off + sizeof(int4) * (size_t)w.max_split, 256);
  w.units_off = off;  off = align_up(off + sizeof(int4) * (size_t)w.max_units, 256);
  w.plse_off = off;   off = align_up(off + sizeof(float) * (size_t)w.max_slots * rc, 256);
  w.po_off = off;     off = align_up(off + sizeof(float) * (size_t)w.max_slots * rc * kDV, 256);
  w.total = off;
  return w;
}

struct SchedArgs {
  const int32_t* seq_lens;
  uint32_t* hdr;
  int4* batch_info;      // (tiles, 0, clamped length, 0)
  int32_t* cta_first;    // first unit of each CTA; [grid] = number of units
  int4* split_list;      // (b, g, pieces, first partial slot) of every cut stream
  int4* units;           // (b, g, tile_begin | tile_end << 16, partial slot or -1)
  int32_t B, s_q, G, max_len, grid;
  int32_t tile;          // keys per tile (128, or 256 for CTA pairs)
  int32_t setup;         // tiles' worth of work charged at the start of every stream
  // fused cache write of the step's new tokens (w_n > 0): done before the schedule
  const uint4* w_latent;
  const uint4* w_rope;
  const int64_t* w_slots;
  uint8_t* w_cache;
  const float* w_kv_scale;
  int64_t w_total_slots;
  int32_t w_n, w_fp8;
  int64_t max_units, max_split, max_slots;
};

struct DecodeArgs {
  CUtensorMap tm_q;      // q as [B][R][576], 64 x RC x 1 boxes, 128-byte swizzle; CTA pairs with
                         // R % 8 == 0: [B][R/8 groups][9 chunks][8 rows][64] (q_whole_rows),
                         // one box of 64 whole rows
  // the cache viewed as [Np*P/8 row groups][9 chunks][8 rows][64 columns]: a box of KC
  // (keys) or 2 (values) chunks x box_rows rows lands in shared memory as
  // [group][chunk][8 rows][64 columns] (bf16: 128-byte swizzle; E4M3: plain)
  CUtensorMap tm_k, tm_v;
  const void* kv_cache;  // [Np][P][576] bf16 or E4M3 bytes
  const int32_t* block_table;
  const int4* batch_info;
  const int4* units;
  const int32_t* cta_first;
  const uint32_t* hdr;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  uint32_t* err;
  const float* kv_scale;
  int32_t s_q, H, R, P, MB, num_pages, causal;
  int32_t box_rows;        // rows of one key/value TMA box: gcd(P, 64)
  float softmax_scale;
  uint64_t wait_limit_ns;  // bound of every pipeline wait (2 s; tests may shorten it)
  int32_t q_whole_rows;    // tm_q loads 64 whole rows per box (see tm_q)
  int32_t test_stall;      // tests only: 1 = the first softmax wait never completes
};

struct CombineArgs {
  const uint32_t* hdr;
  uint32_t* err;           // the device error word (hdr[0])
  const int64_t* w_slots;  // fused cache write: its slots are checked here (w_n > 0)
  int64_t w_total_slots;
  int32_t w_n;
  // the block-table entries the decode read are checked here: [B][MB], the first
  // ceil(L_b / P) of row b (L_b the clamped length in batch_info[b].z)
  const int32_t* block_table;
  const int4* batch_info;
  int32_t B, MB, P, num_pages;
  const int4* split_list;
  const float* part_o;
  const float* part_lse;
  __nv_bfloat16* out;
  float* lse;
  int32_t R, RC;
};

// Launchers (return the launch error).
cudaError_t launch_schedule(const SchedArgs& a, cudaStream_t s);
// CTA-pair decode (rc = 128): grid = 2 * pairs CTAs in clusters of two.
cudaError_t launch_decode_pair(const DecodeArgs& a, bool fp8, int pairs, cudaStream_t s);
cudaError_t decode_pair_prepare(bool fp8);
cudaError_t launch_decode(const DecodeArgs& a, int rc, bool fp8, int grid, cudaStream_t s);
cudaError_t decode_prepare(int rc, bool fp8);   // per-device kernel attributes
int decode_key_chunks_per_slot(int rc, bool fp8);  // chunks in one key TMA box
int decode_value_chunks_per_box(int rc, bool fp8);  // chunks in one value TMA box
cudaError_t launch_combine(const CombineArgs& a, int grid, cudaStream_t s);
cudaError_t launch_cache_write(const void* latent, const void* rope, const int64_t* slots,
                               int32_t n, void* cache, int64_t total_slots, bool fp8,
                               const float* kv_scale, uint32_t* err, cudaStream_t s);

}  // namespace mla
