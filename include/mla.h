/*
 * mla.h — paged Multi-head Latent Attention decode, absorbed-MQA form, for sm_103a.
 *
 * What the library computes
 * -------------------------
 * "[WIP][Attention] FlashAttn MLA" (opening post) runs the decode step of MLA as
 * multi-query attention: after weight absorption, every query head attends over ONE
 * shared latent key/value head. The kernel-test log quoted in "[Attention] Blackwell FP8 MLA
 * support with CUTLASS_MLA backend" (comment by elvischenv) fixes the shapes:
 * h_kv = 1, d = 576 (512 latent + 64 rope) for the scores, dv = 512 for the output,
 * s_q new tokens per sequence, causal, a paged cache, and an FP8 (float8_e4m3fn)
 * cache variant. "[NVIDIA] Add Cutlass MLA backend" (PR body, review thread) adds
 * the block table / block size and the op, ops.cutlass_mla_decode().
 *
 * For sequence b (length L_b = seq_lens[b], which counts the s_q new tokens), new
 * token i and head h:
 *   K[j]  = dequant(kv_cache[block_table[b][j / P]][j % P][0:576]),  j < L_b
 *   V[j]  = K[j][0:512]
 *   s_j   = softmax_scale * dot(q[b][i][h][0:576], K[j]),            j < n_i
 *   out[b][i][h] = sum_j softmax(s)_j V[j];   lse[b][i][h] = ln(sum_j exp(s_j))
 * with n_i = L_b - s_q + 1 + i when causal (the new tokens are the last s_q
 * positions; bottom-right alignment) and n_i = L_b otherwise. Dequantisation is the
 * bf16 value itself, or e4m3(byte) * kv_scale for the FP8 cache (one per-tensor
 * scale). Tokens of the last page beyond L_b and block-table entries beyond
 * ceil(L_b / P) are never used; they may hold anything, NaN included (the prior
 * kernel required the table to be padded; this one does not).
 *
 * Conventions (all entry points)
 * ------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller; the library never
 *   allocates device memory, never frees, and never synchronises the stream.
 * - Layouts are dense row-major as written next to each argument.
 * - Neither outputs nor the workspace need to be zeroed beforehand: every value a
 *   kernel reads from them it wrote earlier in the same call. (The review thread of
 *   "[NVIDIA] Add Cutlass MLA backend" asks whether the prior kernel's output must be
 *   zero-filled by the caller; here uninitialised buffers are fine.)
 * - Host-detectable errors return a negative mla_status and launch nothing.
 *   Errors only the device can see (a block-table entry outside [0, num_pages), a
 *   sequence length outside [s_q, min(max_seq_len, max_blocks_per_seq*page_size)],
 *   with the FP8 cache and 33-64 query rows a query value outside the float16 range,
 *   a stalled pipeline) set bits
 *   of a device error word; mla_decode_check() reads it. Such entries are not
 *   dereferenced out of bounds.
 * - Asynchronous CUDA faults surface at the caller's next synchronisation.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 1

/* A CUDA stream (identical to cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* mla_stream_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,          /* a null pointer, a bad size or a misaligned pointer */
  MLA_ERR_UNSUPPORTED = -2,          /* valid in general but outside this build's limits */
  MLA_ERR_WORKSPACE_TOO_SMALL = -3,
  MLA_ERR_CUDA = -4,                 /* a CUDA runtime call failed (e.g. no device) */
  MLA_ERR_TIMEOUT = -5,              /* device error word: a pipeline wait gave up */
  MLA_ERR_DEVICE_INDEX = -6          /* device error word: a block-table entry, sequence
                                        length, slot or (FP8 cache) query value was out of
                                        range */
} mla_status;

typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype;

/* Device error word bits (see mla_decode_check). */
#define MLA_DEVERR_BLOCK_TABLE   0x1u   /* block_table entry outside [0, num_pages) */
#define MLA_DEVERR_SEQ_LEN       0x2u   /* seq_lens[b] outside the allowed range */
#define MLA_DEVERR_Q_RANGE       0x4u   /* FP8 cache, 33-64 rows: |q| above the float16 range */
#define MLA_DEVERR_TIMEOUT       0x8u   /* a bounded pipeline wait expired */
#define MLA_DEVERR_SLOT          0x10u  /* cache write: slot >= num_pages*page_size */

typedef struct mla_decode_params {
  int32_t batch;               /* B >= 1 */
  int32_t s_q;                 /* new query tokens per sequence, 1..512 */
  int32_t num_heads;           /* H >= 1; s_q * H <= 65536 */
  int32_t page_size;           /* P: a multiple of 8, at most 1024 (else UNSUPPORTED) */
  int32_t num_pages;           /* Np: pages in the pool */
  int32_t max_blocks_per_seq;  /* MB: row stride of block_table */
  int32_t max_seq_len;         /* host-known upper bound on seq_lens[], <= 2^20;
                                  sizes the workspace */
  int32_t kv_dtype;            /* mla_kv_dtype */
  int32_t causal;              /* 0 or 1; only matters when s_q > 1 */
} mla_decode_params;

/* Workspace bytes mla_decode needs for these parameters on a GPU with `num_sms`
 * multiprocessors (num_sms <= 0: the current device's count). 0 on invalid params.
 * The size does not depend on the contents of seq_lens. */
size_t mla_decode_workspace_size(const mla_decode_params* p, int32_t num_sms);

/* Paged absorbed-MQA decode (see the top of this file).
 *   q            [B, s_q, H, 576] bf16, 16-byte aligned
 *   kv_cache     [Np, P, 576]  bf16 (kv_dtype BF16) or e4m3fn bytes (FP8), 16-byte aligned
 *   block_table  [B, MB] int32: physical page of each logical page
 *   seq_lens     [B] int32: tokens per sequence including the s_q new ones
 *   softmax_scale  multiplies q.K (e.g. 1/sqrt(192) for DeepSeek's 128+64 head dim)
 *   kv_scale     device float scalar; the FP8 dequantisation scale (ignored, may be
 *                NULL, for a bf16 cache)
 *   out          [B, s_q, H, 512] bf16 (written)
 *   lse          [B, s_q, H] float32, natural log (written)
 *   workspace    >= mla_decode_workspace_size(p, 0) bytes, 256-byte aligned; its first
 *                4 bytes hold the device error word after the call
 * Launches a split scheduler, the split-KV decode kernel and the LSE combine on
 * `stream`, in that order; returns without synchronising. */
mla_status mla_decode(const mla_decode_params* p, const void* q, const void* kv_cache,
                      const int32_t* block_table, const int32_t* seq_lens,
                      float softmax_scale, const float* kv_scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* mla_cache_write of a decode step's new tokens followed by mla_decode, in one launch
 * chain ("[Attention] Blackwell FP8 MLA support with CUTLASS_MLA backend", Purpose: the
 * FP8 cache the decode reads; the step appends each sequence's s_q new latent rows and
 * attends over them). Arguments as mla_cache_write (latent, rope, slot_mapping,
 * num_tokens; the cache geometry and kv_dtype come from `p`) and as mla_decode. The new
 * rows are written by extra CTAs of the split scheduler's launch while its first CTA
 * computes the schedule, one launch fewer than the two calls (beyond 2^17 tokens the
 * cache-write kernel runs ahead of the scheduler instead); the decode reads the cache
 * only after that launch has completed. seq_lens counts the new tokens, whose slots lie
 * in the sequences' pages. A slot outside the pool is skipped and reported as
 * MLA_DEVERR_SLOT through mla_decode_check. */
mla_status mla_decode_with_cache_write(const mla_decode_params* p, const void* latent, const void* rope,
                                       const int64_t* slot_mapping, int32_t num_tokens, const void* q,
                                       void* kv_cache, const int32_t* block_table,
                                       const int32_t* seq_lens, float softmax_scale,
                                       const float* kv_scale, void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, mla_stream_t stream);

/* Synchronises `stream`, then reads the device error word left in `workspace` by the
 * last mla_decode on it: MLA_OK, MLA_ERR_DEVICE_INDEX, MLA_ERR_TIMEOUT, or
 * MLA_ERR_CUDA. If `bits` is not NULL it receives the raw MLA_DEVERR_* bits. */
mla_status mla_decode_check(const void* workspace, mla_stream_t stream, uint32_t* bits);

/* Paged cache write ("[Attention] Blackwell FP8 MLA support with CUTLASS_MLA
 * backend", Purpose: the FP8 KV cache). Token t's row concat(latent[t], rope[t]) is
 * stored at slot s = slot_mapping[t], i.e. page s / P, row s % P.
 *   latent        [N, 512] bf16;  rope [N, 64] bf16 (16-byte aligned rows)
 *   slot_mapping  [N] int64; s < 0 marks a padding token (skipped)
 *   kv_cache      [Np, P, 576] bf16 or e4m3fn bytes
 *   kv_scale      device float scalar (FP8 only): byte = e4m3_rne_satfinite(x / kv_scale)
 *                 with x / kv_scale an IEEE float32 division; bf16: the bits are copied
 *   device_error  optional device uint32; MLA_DEVERR_SLOT is OR-ed into it for a slot
 *                 >= Np * P (that token is skipped). May be NULL.
 * One launch on `stream`; no synchronisation. */
mla_status mla_cache_write(const void* latent, const void* rope, const int64_t* slot_mapping,
                           int32_t num_tokens, void* kv_cache, int32_t num_pages,
                           int32_t page_size, int32_t kv_dtype, const float* kv_scale,
                           uint32_t* device_error, mla_stream_t stream);

/* No-allocation variant of mla_decode. This entry point has no counterpart in the
 * pages; it exists for callers that cannot allocate device memory — for example a
 * plugin inside an inference engine whose interface passes only inputs and outputs, or
 * a runtime that owns all device memory through its own allocator and forbids (or
 * cannot afford the implicit device synchronisation of) a cudaMalloc.
 * Same arguments and results as mla_decode without the workspace: the scratch memory
 * lives in a static device array of the library, MLA_NOALLOC_SCRATCH_BYTES long, that
 * every GPU which loads the library holds until the process exits. No cudaMalloc,
 * cudaFree or other allocating call is made.
 * - Returns MLA_ERR_WORKSPACE_TOO_SMALL, launching nothing, when the parameters need
 *   more scratch than that (mla_decode_workspace_size(p, 0) > MLA_NOALLOC_SCRATCH_BYTES).
 *   On a 152-SM GB300 that admits up to 32 query rows per sequence (s_q * H <= 32, e.g.
 *   16 or 32 heads at s_q = 1); 64 or more rows need more split scratch and are refused.
 * - The first call on a device looks up the array's device address (with that device
 *   current) and caches it; make that first call before any stream capture.
 * - All calls share the one array, which keeps the last call's contents (nothing in it
 *   needs clearing: each call writes every scratch word it reads). Calls that overlap
 *   on the GPU (other streams, other threads) race on it: serialise them. */
#define MLA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
mla_status mla_decode_noalloc(const mla_decode_params* p, const void* q, const void* kv_cache,
                              const int32_t* block_table, const int32_t* seq_lens,
                              float softmax_scale, const float* kv_scale, void* out, float* lse,
                              mla_stream_t stream);

/* mla_decode_check for mla_decode_noalloc: synchronises `stream` and reads the device error
 * word that the last no-allocation call left in the library's static scratch array (same
 * results and `bits` as mla_decode_check). Allocates nothing. */
mla_status mla_decode_noalloc_check(mla_stream_t stream, uint32_t* bits);

/* Decode-kernel timing, for benchmarks and tests. After mla_profile_begin(n), each of the
 * next n mla_decode / mla_decode_noalloc calls in this process records a CUDA event on
 * its stream immediately before and immediately after its decode-kernel launch. The
 * events belong to the library and are created on the device current at
 * mla_profile_begin; the timed calls must run on that device. The event between the
 * scheduler and the decode kernel also makes the decode kernel wait until the scheduler
 * has finished (no overlap of its set-up), so each interval is the decode kernel alone.
 * mla_profile_end waits for the recorded events, stores the summed decode-kernel time
 * in milliseconds in *total_ms and the number of timed launches in *launches, and stops
 * recording (with no mla_profile_begin before it: 0 and 0). Not thread safe: one
 * profiling window per process at a time.
 * Errors: MLA_ERR_INVALID_ARG for max_launches outside [1, 4096] or a NULL output;
 * MLA_ERR_CUDA when an event cannot be created, recorded or read. */
mla_status mla_profile_begin(int32_t max_launches);
mla_status mla_profile_end(double* total_ms, int32_t* launches);

/* Test support (not for production use; not thread safe). Every pipeline wait inside the
 * decode kernels is bounded: after `wait_limit_ns` (0 restores the default, 2 s) it gives
 * up, sets MLA_DEVERR_TIMEOUT in the device error word, and the kernel drains its copies
 * and MMAs and exits, leaving the CUDA context usable. With stall = 1 the first softmax
 * wait of every CTA waits on a barrier nothing arrives on, so that the bound is reached
 * without any fault; stall = 0 restores normal operation. Applies to the decode calls
 * launched after it. Errors: MLA_ERR_INVALID_ARG for a stall value other than 0 or 1. */
mla_status mla_test_set_hooks(uint64_t wait_limit_ns, int32_t stall);

/* Static text for a status code. */
const char* mla_status_string(int32_t status);

/* MLA_ABI_VERSION of the loaded library. */
int32_t mla_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
