// mla_api.cu — the C ABI (include/mla.h): argument checks, workspace layout, TMA
// descriptors and the launch sequence  schedule -> decode -> combine  on one stream.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>
#include <cudaTypedefs.h>
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "../../include/mla.h"

#define MLA_EXPORT extern "C" __attribute__((visibility("default")))

namespace mla {
namespace {

constexpr int kMaxDevices = 64;

std::atomic<int> g_num_sms[kMaxDevices];
std::atomic<uint32_t> g_prepared[kMaxDevices];   // bit per decode variant
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// decode-kernel timing window (mla_profile_begin / mla_profile_end)
struct ProfileWindow {
  std::vector<cudaEvent_t> ev;   // 2 per launch: before, after
  int cap = 0, next = 0;
  bool on = false;
};
ProfileWindow g_prof;
constexpr int kMaxProfiledLaunches = 4096;

// test hooks (mla_test_set_hooks): the wait bound passed to the kernels and the stall flag
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
std::atomic<int32_t> g_test_stall{0};

int variant_bit(int rc, bool fp8) {
  return (rc == 16 ? 0 : rc == 32 ? 2 : rc == 64 ? 4 : 6) + (fp8 ? 1 : 0);
}

cudaError_t current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
  return cudaSuccess;
}

int sm_count(int dev) {
  int n = g_num_sms[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return -1;
  g_num_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool get_encoder() {
  if (g_encode) return true;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

mla_status check_params(const mla_decode_params* p) {
  if (p == nullptr) return MLA_ERR_INVALID_ARG;
  if (p->batch < 1 || p->s_q < 1 || p->num_heads < 1 || p->page_size < 1 || p->num_pages < 1 ||
      p->max_blocks_per_seq < 1 || p->max_seq_len < 1)
    return MLA_ERR_INVALID_ARG;
  if (p->kv_dtype != MLA_KV_BF16 && p->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return MLA_ERR_INVALID_ARG;
  if (p->max_seq_len < p->s_q) return MLA_ERR_INVALID_ARG;
  if (p->page_size % 8 != 0 || p->page_size > 1024) return MLA_ERR_UNSUPPORTED;
  if (p->s_q > kMaxSq || (int64_t)p->s_q * p->num_heads > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (p->batch > kMaxBatch || p->max_seq_len > kMaxSeqLen) return MLA_ERR_UNSUPPORTED;
  if ((int64_t)p->num_pages * p->page_size >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
  if ((int64_t)p->max_blocks_per_seq * p->page_size < p->s_q) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

// The cache as [rows / 8 groups][9 chunks][8 rows][64 elements] (strides 8 rows, one
// chunk, one row): a box of `chunks` chunks x box_rows / 8 groups lands in shared memory
// as [group][chunk][8 rows][64 elements]. bf16 rows (128 B) are 128-byte swizzled for
// the MMA. E4M3 rows (64 B) with sw64 are 64-byte swizzled: the layout of the 8-bit MMA
// operands (CTA pairs), and one in which 32 threads reading one key row each hit distinct
// banks (the converting threads of the single-CTA kernel); its E4M3 value rows are plain.
bool encode_kv_map(CUtensorMap* m, const void* cache, int64_t rows, uint32_t chunks, uint32_t box_rows,
                   bool fp8, bool sw64) {
  const cuuint64_t es = fp8 ? 1 : 2;
  cuuint64_t dims[4] = {64, 8, 9, (cuuint64_t)(rows / 8)};
  cuuint64_t strides[3] = {kDQK * es, 64 * es, kDQK * es * 8};
  cuuint32_t box[4] = {64, 8, chunks, box_rows / 8};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                        const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        !fp8 ? CU_TENSOR_MAP_SWIZZLE_128B
                             : sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// q as [B][R/8 groups][9 chunks][8 rows][64 elements]: a box of 8 groups x 9 chunks is 64
// whole 1152-byte rows (one contiguous piece each, the cheapest for TMA), landing as
// [group][chunk][8 rows][64] with 128-byte swizzle. Needs R % 8 == 0.
bool encode_q_rows_map(CUtensorMap* m, const void* q, int B, int R) {
  cuuint64_t dims[5] = {64, 8, 9, (cuuint64_t)(R / 8), (cuuint64_t)B};
  cuuint64_t strides[4] = {(cuuint64_t)kDQK * 2, 128, (cuuint64_t)kDQK * 2 * 8, (cuuint64_t)kDQK * 2 * R};
  cuuint32_t box[5] = {64, 8, 9, 8, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(q), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap* m, const void* q, int B, int R, int rc) {
  cuuint64_t dims[3] = {(cuuint64_t)kDQK, (cuuint64_t)R, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)kDQK * 2, (cuuint64_t)kDQK * 2 * R};
  cuuint32_t box[3] = {64, (cuuint32_t)rc, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace mla

using namespace mla;

MLA_EXPORT int32_t mla_abi_version(void) { return MLA_ABI_VERSION; }

MLA_EXPORT const char* mla_status_string(int32_t s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MLA_ERR_DEVICE_INDEX: return "device-side index or length out of range";
    default: return "unknown status";
  }
}

MLA_EXPORT size_t mla_decode_workspace_size(const mla_decode_params* p, int32_t num_sms) {
  if (check_params(p) != MLA_OK) return 0;
  if (num_sms <= 0) {
    int dev;
    if (current_device(&dev) != cudaSuccess) return 0;
    num_sms = sm_count(dev);
    if (num_sms <= 0) return 0;
  }
  const Plan plan = make_plan(p->s_q * p->num_heads, p->kv_dtype == MLA_KV_FP8_E4M3);
  return ws_layout(p->batch, plan, plan_workers(plan, num_sms)).total;
}

namespace mla {
namespace {
// The step's new tokens for the fused cache write (num == 0: none).
struct FusedWrite {
  const void* latent;
  const void* rope;
  const int64_t* slots;
  int32_t num;
};
}  // namespace
}  // namespace mla

static mla_status decode_impl(const mla_decode_params* p, const void* q, const void* kv_cache,
                              const int32_t* block_table, const int32_t* seq_lens, float softmax_scale,
                              const float* kv_scale, void* out, float* lse, void* workspace,
                              size_t workspace_bytes, mla_stream_t stream, const FusedWrite& fw) {
  mla_status st = check_params(p);
  if (st != MLA_OK) return st;
  const bool fp8 = p->kv_dtype == MLA_KV_FP8_E4M3;
  if (!q || !kv_cache || !block_table || !seq_lens || !out || !lse || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (fp8 && !kv_scale) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(workspace, 256))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale) || softmax_scale > 3.0e38f || softmax_scale < -3.0e38f)
    return MLA_ERR_INVALID_ARG;

  int dev;
  if (current_device(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  const int nsm = sm_count(dev);
  if (nsm <= 0) return MLA_ERR_CUDA;
  const int B = p->batch, R = p->s_q * p->num_heads;
  const Plan plan = make_plan(R, fp8);
  const int rc = plan.rc, G = plan.G;
  const int grid = plan_workers(plan, nsm);
  if (grid < 1) return MLA_ERR_UNSUPPORTED;
  const WsLayout w = ws_layout(B, plan, grid);
  if (workspace_bytes < w.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!get_encoder()) return MLA_ERR_CUDA;

  const uint32_t bit = 1u << variant_bit(rc, fp8);
  if (!(g_prepared[dev].load() & bit)) {
    if ((plan.pair ? decode_pair_prepare(fp8) : decode_prepare(rc, fp8)) != cudaSuccess) return MLA_ERR_CUDA;
    g_prepared[dev].fetch_or(bit);
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* hdr = reinterpret_cast<uint32_t*>(ws);
  int4* batch_info = reinterpret_cast<int4*>(ws + w.batch_off);
  int32_t* cta_first = reinterpret_cast<int32_t*>(ws + w.cta_off);
  int4* split_list = reinterpret_cast<int4*>(ws + w.split_off);
  int4* units = reinterpret_cast<int4*>(ws + w.units_off);
  float* plse = reinterpret_cast<float*>(ws + w.plse_off);
  float* po = reinterpret_cast<float*>(ws + w.po_off);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  SchedArgs sa{};
  sa.seq_lens = seq_lens;
  sa.hdr = hdr;
  sa.batch_info = batch_info;
  sa.cta_first = cta_first;
  sa.split_list = split_list;
  sa.units = units;
  sa.B = B;
  sa.s_q = p->s_q;
  sa.G = G;
  const int64_t cap = (int64_t)p->max_blocks_per_seq * p->page_size;
  sa.max_len = (int)(cap < p->max_seq_len ? cap : p->max_seq_len);
  sa.grid = grid;
  sa.tile = plan.tile;
  // a unit's set-up (its q, the pipeline's refill, its epilogue) is charged to the CTA that
  // starts the stream, in tiles of streaming: measured best at 2 for bf16 CTA pairs, 3 for
  // FP8 pairs and 4 for the FP8 cache with up to 64 rows; with bf16 and up to 64 rows a unit
  // change costs little (0)
  sa.setup = plan.pair ? (fp8 ? 3 : 2) : fp8 ? 4 : 0;
  sa.max_units = w.max_units;
  sa.max_split = w.max_split;
  sa.max_slots = w.max_slots;
  if (fw.num > 0) {
    // the new tokens' rows go into the cache ahead of the decode: CTAs of the scheduler's
    // launch write them next to the schedule computation (for very large writes, the
    // cache-write kernel runs ahead of the scheduler instead)
    const int64_t total_slots = (int64_t)p->num_pages * p->page_size;
    if (fw.num <= kMaxFusedWriteTokens) {
      sa.w_latent = static_cast<const uint4*>(fw.latent);
      sa.w_rope = static_cast<const uint4*>(fw.rope);
      sa.w_slots = fw.slots;
      sa.w_cache = static_cast<uint8_t*>(const_cast<void*>(kv_cache));
      sa.w_kv_scale = kv_scale;
      sa.w_total_slots = total_slots;
      sa.w_n = fw.num;
      sa.w_fp8 = fp8 ? 1 : 0;
    } else if (launch_cache_write(fw.latent, fw.rope, fw.slots, fw.num, const_cast<void*>(kv_cache), total_slots, fp8,
                                  kv_scale, nullptr, s) != cudaSuccess) {
      return MLA_ERR_CUDA;
    }
  }
  if (launch_schedule(sa, s) != cudaSuccess) return MLA_ERR_CUDA;

  DecodeArgs da;
  std::memset(&da, 0, sizeof(da));
  // key / value boxes of gcd(P, 64) rows never straddle a page
  const int box_rows = std::min(64, p->page_size & -p->page_size);
  // a CTA of a pair holds 64 of its unit's 128 rows (as whole rows when R % 8 == 0)
  da.q_whole_rows = plan.pair && R % 8 == 0 ? 1 : 0;
  if (da.q_whole_rows ? !encode_q_rows_map(&da.tm_q, q, B, R) : !encode_q_map(&da.tm_q, q, B, R, plan.pair ? 64 : rc))
    return MLA_ERR_INVALID_ARG;
  {
    const int64_t rows = (int64_t)p->num_pages * p->page_size;
    // chunks per key / value box: a pair loads 256-byte pieces of each bf16 key row (2
    // chunks) or whole E4M3 key rows (9 chunks), and 4 adjacent chunks of each value row
    const uint32_t kc = plan.pair ? (fp8 ? 9u : 2u) : (uint32_t)decode_key_chunks_per_slot(rc, fp8);
    const uint32_t vc = plan.pair ? 4u : (uint32_t)decode_value_chunks_per_box(rc, fp8);
    // E4M3 keys and values are 64-byte swizzled: the MMAs read them as they land
    if (!encode_kv_map(&da.tm_k, kv_cache, rows, kc, (uint32_t)box_rows, fp8, true) ||
        !encode_kv_map(&da.tm_v, kv_cache, rows, vc, (uint32_t)box_rows, fp8, true))
      return MLA_ERR_INVALID_ARG;
  }
  da.kv_cache = kv_cache;
  da.block_table = block_table;
  da.batch_info = batch_info;
  da.units = units;
  da.cta_first = cta_first;
  da.hdr = hdr;
  da.out = static_cast<__nv_bfloat16*>(out);
  da.lse = lse;
  da.part_o = po;
  da.part_lse = plse;
  da.err = hdr;
  da.kv_scale = kv_scale;
  da.s_q = p->s_q;
  da.H = p->num_heads;
  da.R = R;
  da.P = p->page_size;
  da.box_rows = box_rows;
  da.MB = p->max_blocks_per_seq;
  da.num_pages = p->num_pages;
  da.causal = p->causal;
  da.softmax_scale = softmax_scale;
  da.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  da.test_stall = g_test_stall.load(std::memory_order_relaxed);
  const bool timed = g_prof.on && g_prof.next < g_prof.cap;
  if (timed && cudaEventRecord(g_prof.ev[2 * g_prof.next], s) != cudaSuccess) return MLA_ERR_CUDA;
  const cudaError_t le = plan.pair ? launch_decode_pair(da, fp8, grid, s) : launch_decode(da, rc, fp8, grid, s);
  if (le != cudaSuccess) return MLA_ERR_CUDA;
  if (timed) {
    if (cudaEventRecord(g_prof.ev[2 * g_prof.next + 1], s) != cudaSuccess) return MLA_ERR_CUDA;
    ++g_prof.next;
  }

  CombineArgs ca{};
  ca.hdr = hdr;
  ca.err = hdr;
  ca.w_slots = fw.num > 0 ? fw.slots : nullptr;
  ca.w_n = fw.num;
  ca.w_total_slots = (int64_t)p->num_pages * p->page_size;
  ca.block_table = block_table;
  ca.batch_info = batch_info;
  ca.B = p->batch;
  ca.MB = p->max_blocks_per_seq;
  ca.P = p->page_size;
  ca.num_pages = p->num_pages;
  ca.split_list = split_list;
  ca.part_o = po;
  ca.part_lse = plse;
  ca.out = static_cast<__nv_bfloat16*>(out);
  ca.lse = lse;
  ca.R = R;
  ca.RC = rc;
  // up to 2 * workers cut streams x RC rows: 8 * #SM blocks of 8 warps give every (stream,
  // row) task its own warp for RC <= 32 and at most two rounds for RC = 64 or 128 (the
  // combine is a few dependent global loads per task: latency, not bandwidth)
  if (launch_combine(ca, 8 * nsm, s) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

MLA_EXPORT mla_status mla_test_set_hooks(uint64_t wait_limit_ns, int32_t stall) {
  if (stall != 0 && stall != 1) return MLA_ERR_INVALID_ARG;
  mla::g_wait_limit_ns.store(wait_limit_ns == 0 ? mla::kWaitLimitNs : wait_limit_ns);
  mla::g_test_stall.store(stall);
  return MLA_OK;
}

MLA_EXPORT mla_status mla_decode(const mla_decode_params* p, const void* q, const void* kv_cache,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 float softmax_scale, const float* kv_scale, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  return decode_impl(p, q, kv_cache, block_table, seq_lens, softmax_scale, kv_scale, out, lse, workspace,
                     workspace_bytes, stream, FusedWrite{nullptr, nullptr, nullptr, 0});
}

MLA_EXPORT mla_status mla_decode_with_cache_write(const mla_decode_params* p, const void* latent,
                                                  const void* rope, const int64_t* slot_mapping,
                                                  int32_t num_tokens, const void* q, void* kv_cache,
                                                  const int32_t* block_table, const int32_t* seq_lens,
                                                  float softmax_scale, const float* kv_scale, void* out,
                                                  float* lse, void* workspace, size_t workspace_bytes,
                                                  mla_stream_t stream) {
  if (num_tokens < 0) return MLA_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!latent || !rope || !slot_mapping)) return MLA_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!aligned(latent, 16) || !aligned(rope, 16) || !aligned(slot_mapping, 8)))
    return MLA_ERR_INVALID_ARG;
  return decode_impl(p, q, kv_cache, block_table, seq_lens, softmax_scale, kv_scale, out, lse, workspace,
                     workspace_bytes, stream, FusedWrite{latent, rope, slot_mapping, num_tokens});
}

MLA_EXPORT mla_status mla_profile_begin(int32_t max_launches) {
  using mla::g_prof;
  if (max_launches < 1 || max_launches > mla::kMaxProfiledLaunches) return MLA_ERR_INVALID_ARG;
  while ((int)g_prof.ev.size() < 2 * max_launches) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return MLA_ERR_CUDA;
    g_prof.ev.push_back(e);
  }
  g_prof.cap = max_launches;
  g_prof.next = 0;
  g_prof.on = true;
  return MLA_OK;
}

MLA_EXPORT mla_status mla_profile_end(double* total_ms, int32_t* launches) {
  using mla::g_prof;
  if (total_ms == nullptr || launches == nullptr) return MLA_ERR_INVALID_ARG;
  const int n = g_prof.on ? g_prof.next : 0;
  g_prof.on = false;
  double sum = 0.0;
  for (int i = 0; i < n; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess)
      return MLA_ERR_CUDA;
    sum += ms;
  }
  *total_ms = sum;
  *launches = n;
  return MLA_OK;
}

MLA_EXPORT mla_status mla_decode_check(const void* workspace, mla_stream_t stream, uint32_t* bits) {
  if (workspace == nullptr) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (bits) *bits = word;
  if (word & MLA_DEVERR_TIMEOUT) return MLA_ERR_TIMEOUT;
  if (word) return MLA_ERR_DEVICE_INDEX;
  return MLA_OK;
}

MLA_EXPORT mla_status mla_cache_write(const void* latent, const void* rope,
                                      const int64_t* slot_mapping, int32_t num_tokens,
                                      void* kv_cache, int32_t num_pages, int32_t page_size,
                                      int32_t kv_dtype, const float* kv_scale,
                                      uint32_t* device_error, mla_stream_t stream) {
  if (num_tokens < 0 || num_pages < 1 || page_size < 1) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  const bool fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  if (num_tokens == 0) return MLA_OK;
  if (!latent || !rope || !slot_mapping || !kv_cache) return MLA_ERR_INVALID_ARG;
  if (fp8 && !kv_scale) return MLA_ERR_INVALID_ARG;
  if (!aligned(latent, 16) || !aligned(rope, 16) || !aligned(kv_cache, 16) ||
      !aligned(slot_mapping, 8) || (device_error && !aligned(device_error, 4)))
    return MLA_ERR_INVALID_ARG;
  const int64_t total = (int64_t)num_pages * page_size;
  if (launch_cache_write(latent, rope, slot_mapping, num_tokens, kv_cache, total, fp8, kv_scale,
                         device_error, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
