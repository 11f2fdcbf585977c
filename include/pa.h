/*
 * pa.h - C ABI of libpagedattn: paged single-query decode attention and the
 * two cache operations around it, for NVIDIA GB300 (sm_103a).
 *
 * Sources restated (page title, then section / equation):
 *  [P1] "論文解説: Efficient Memory Management for Large Language Model Serving
 *       with PagedAttention" (0h-n0.github.io): "PagedAttentionのメモリ管理",
 *       "Attention計算", "Copy-on-Write（CoW）によるメモリ共有",
 *       "GPUカーネル最適化".
 *  [P2] "KVキャッシュとPagedAttention — 推論メモリのすべて" (youngju.dev):
 *       "PagedAttention: OS仮想メモリ式の管理", "prefix共有とcopy-on-write",
 *       "KV量子化: FP8とINT8", "GQAとMQA".
 *  [P3] "PagedAttention" notes (dihengye.cn): "分块 Attention 计算".
 *  [P4] "メモリ予算内での言語モデルのサービング" (auturnal.com): equation (4).
 *
 * Conventions shared by every call
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *    library allocates nothing and keeps no reference after the call returns.
 *    The caller owns every buffer.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and enqueues its work on the current device.
 *  - Host-side validation happens before anything is enqueued: a negative
 *    pa_status is returned and nothing runs.  PA_ERR_CUDA reports a failed
 *    launch or CUDA runtime call.
 *  - Device-side checks never trap.  Out-of-range block ids, slots, pairs or
 *    sequence lengths are skipped and recorded in a per-device error word
 *    that pa_get_device_error() reads and clears.
 *  - KV cache layout: two separate pools k_cache and v_cache, each
 *    [num_blocks][num_kv_heads][block_size][head_dim], row-major.  One
 *    (block, head) tile is block_size*head_dim contiguous elements.
 *    Token position p of a sequence lives in physical block
 *    block_tables[s][p / block_size], row p % block_size  ([P1]
 *    "PagedAttentionのメモリ管理": the block table maps logical blocks to
 *    physical blocks of B tokens).
 *  - Supported shapes: head_dim in {64, 128} for 16-bit caches, 128 for the
 *    8-bit (FP8, INT8) caches, which also take at most 256 KV heads; block_size a power of two from 8 to 1024 (16
 *    and 32 are the usual sizes); num_heads = G * num_kv_heads with
 *    1 <= G <= 8; with q_len queries per sequence (pa_decode_ex),
 *    q_len * G <= 64.
 */
#ifndef PAGEDATTN_PA_H
#define PAGEDATTN_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_F32 = 0,
  PA_F16 = 1,
  PA_BF16 = 2,
  PA_FP8_E4M3 = 3, /* OCP E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa; max 448 */
  PA_INT8 = 4      /* signed 8-bit code with a per-KV-head scale and zero point:
                      value = (code - zero_point) * scale */
} pa_dtype;

typedef enum {
  PA_OK = 0,
  PA_ERR_NULL = -1,        /* a required pointer is NULL */
  PA_ERR_SHAPE = -2,       /* inconsistent or out-of-range sizes */
  PA_ERR_DTYPE = -3,       /* dtype combination not accepted */
  PA_ERR_UNSUPPORTED = -4, /* valid request outside the compiled variants */
  PA_ERR_WORKSPACE = -5,   /* workspace missing or smaller than required */
  PA_ERR_CUDA = -6,        /* CUDA runtime / launch failure */
  PA_ERR_ALIGN = -7        /* a pointer or stride breaks the 16-byte rule */
} pa_status;

/* Bits of the per-device error word (pa_get_device_error). */
#define PA_DEVERR_BLOCK_ID 1u /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_SLOT 2u     /* slot outside [0, num_blocks*block_size) */
#define PA_DEVERR_SEQ_LEN 4u  /* seq_len < 0 or > max_blocks_per_seq*block_size */
#define PA_DEVERR_TIMEOUT 8u  /* a bounded wait on an async copy gave up */
#define PA_DEVERR_PAIR 16u    /* copy_blocks id outside [0, num_blocks) */
#define PA_DEVERR_INTERNAL 32u /* a sizing invariant of the library failed (a bug; the result is wrong) */

/*
 * pa_decode_workspace_bytes
 *   Bytes of device workspace that pa_decode needs for these sizes on the
 *   CURRENT device (the split-K partial records depend on the device's SM
 *   count).  Returns 0 when the call needs no workspace (single pass) and
 *   (size_t)-1 when the sizes are rejected or no device is usable.
 *   The workspace must be zero-filled once before its first use; every
 *   completed pa_decode leaves it ready for the next call (a call that set
 *   PA_DEVERR_TIMEOUT may leave counters behind: zero it again after one).
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_blocks_per_seq, int partition_size,
                                 pa_dtype kv_dtype);

/*
 * pa_decode - one decode step of paged attention.
 *
 * For every sequence s and query head h (KV head kvh = h / G, G = num_heads /
 * num_kv_heads, [P2] "GQAとMQA"):
 *     out[s][h] = softmax(scale * K_s q[s][h]) V_s
 * where K_s, V_s are the seq_lens[s] rows of KV head kvh gathered through
 * block_tables[s] ([P1] "Attention計算"; [P3] "分块 Attention 计算").  The
 * kernel reads the blocks one by one and merges them with the online-softmax
 * recurrence ([P4] eq. (4)); long sequences are split across warps and the
 * per-split states (m, l, acc) are merged with the same recurrence by the
 * last split to finish ("split-K").  seq_lens[s] == 0 gives out[s] = 0.
 * FP8 caches ([P2] "KV量子化") are dequantised in registers as
 * float(e4m3) * k_scale[kvh] (resp. v_scale[kvh]).
 * With an 8-bit cache (FP8, or INT8 through pa_decode_ex) the two products
 * run with f16 operands (the widened cache values are exact in f16) and fp32
 * accumulation.  A bf16 query group (the G query rows of one sequence and KV
 * head) is first multiplied by the power of two 2^e that puts its largest
 * |q| in [2^14, 2^15), and the scores by 2^-e: no value overflows f16, and
 * every element within a factor 2^28 of the group's largest is represented
 * exactly (smaller elements may round as f16 subnormals, an absolute error
 * below 2^-38 times the group's largest |q|).  Any finite bf16 query is
 * accepted.
 *
 *   out            [num_seqs][num_heads][head_dim], out_dtype F32/F16/BF16
 *   q              [num_seqs][num_heads][head_dim] at q_stride elements per
 *                  sequence (q_stride >= num_heads*head_dim), q_dtype F16/BF16;
 *                  16-byte aligned base, q_stride*sizeof(q) % 16 == 0
 *   k_cache/v_cache  pools as above, kv_dtype F16/BF16 (== q_dtype) or
 *                  FP8_E4M3; 16-byte aligned; num_blocks blocks each
 *   k_scale/v_scale  float32 [num_kv_heads]; required for FP8, else ignored
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]; entries beyond
 *                  ceil(seq_lens[s]/block_size) are never read
 *   seq_lens       int32 [num_seqs]
 *   scale          softmax scale (e.g. 1/sqrt(head_dim)), float32
 *   partition_size 0   = balanced split: equal shares of all KV blocks to
 *                        every resident warp (recommended);
 *                  P>0 = fixed partitions of P tokens (P % block_size == 0),
 *                        one warp each; P >= max_blocks_per_seq*block_size
 *                        is a single pass that needs no workspace.
 *   workspace      device buffer of >= pa_decode_workspace_bytes(...) bytes,
 *                  zero-filled before first use; NULL allowed when 0 bytes
 *                  are required.  Calls that share a workspace must not
 *                  overlap on the GPU.
 *   stream         cudaStream_t
 */
int pa_decode(void* out, pa_dtype out_dtype,
              const void* q, pa_dtype q_dtype, int64_t q_stride,
              const void* k_cache, const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
              const float* k_scale, const float* v_scale,
              const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* seq_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim,
              float scale, int block_size, int partition_size,
              void* workspace, size_t workspace_bytes,
              void* stream);

/*
 * pa_decode_ex - pa_decode with options: variants of the decode step that a
 * serving system adds on top of the plain one.
 *
 * Same arguments and semantics as pa_decode, plus `opt` (NULL = all options
 * off, i.e. exactly pa_decode).  The caller sets opt->struct_size to
 * sizeof(pa_decode_options) as it was compiled; fields beyond that size are
 * taken as 0, so older callers keep working when fields are added.
 *
 *   window   > 0: sliding-window decode.  The query of sequence s, at
 *            position seq_lens[s]-1, attends to positions
 *            max(0, seq_lens[s]-window) .. seq_lens[s]-1 only, and only the
 *            blocks holding them are read (the "局限性与未来工作" list of the
 *            dihengye.cn notes names sliding-window attention as a limitation
 *            of the paged kernel; this is its plainest reading).  0 = the
 *            whole sequence.  Negative values are rejected (PA_ERR_SHAPE).
 *   k_zero_point / v_zero_point
 *            int32 [num_kv_heads] device arrays, values in [-128, 127];
 *            required for kv_dtype PA_INT8 (k_scale / v_scale are then the
 *            INT8 scales), ignored otherwise ([P2] "KV量子化: FP8とINT8":
 *            INT8 KV needs a scale and a zero point).
 *   k_new / v_new  (fused append; NULL = off)
 *            rows [num_seqs][num_kv_heads][head_dim] of every sequence's
 *            newest position seq_lens[s]-1, new_stride elements apart per
 *            sequence, new_dtype F16/BF16 (== kv_dtype for 16-bit caches).
 *            The call first stores them into the slot that position maps to
 *            through block_tables (quantised with k_inv_scale / v_inv_scale,
 *            and the zero points for INT8, exactly as pa_reshape_and_cache
 *            does) and attends over all seq_lens[s] rows including them: one
 *            launch for the cache write and the decode of a step ([P2]
 *            "PagedAttention: OS仮想メモリ式の管理": a new token's rows go into
 *            the slot of its position).  16-byte aligned bases,
 *            new_stride*2 % 16 == 0.  Sequences with seq_lens[s] == 0 write
 *            nothing.  Needs q_len 1.
 *   q_len    queries per sequence (0 or 1: one).  With q_len = L the L
 *            newest positions T-L .. T-1 of each sequence (T = seq_lens[s],
 *            rows already in the cache) are queries: q and out are
 *            [num_seqs][L][num_heads][head_dim] (q at q_stride >= L*num_heads*
 *            head_dim elements per sequence, out packed) and query i attends
 *            to positions up to its own, T-L+i (with a window: the last
 *            `window` of them).  A query whose position is negative (T < L)
 *            gets out = 0.  L * (num_heads / num_kv_heads) <= 64, else
 *            PA_ERR_UNSUPPORTED (up to 16 (query, head) rows are served by
 *            one consumer warp per K/V stage, more by 2-4 warps that share
 *            each stage, 16 rows each).  This is the verification step of
 *            speculative decoding, which the explainer names alongside paged
 *            KV memory.
 *   pdl      nonzero: launch with programmatic dependent launch, so that the
 *            decode's set-up overlaps the kernel launched just before it on
 *            `stream` (typically pa_reshape_and_cache of the same step, whose
 *            kernel lets its dependents start at once).  During that overlap
 *            the decode reads seq_lens and block_tables only; it reads q, the
 *            caches, the scales and the new rows, and writes out, the cache
 *            and the workspace, only after that kernel has finished.  So with
 *            pdl on, seq_lens and block_tables must not be written by the
 *            kernel launched just before this call (host copies and earlier
 *            kernels are fine).  0: an ordinary launch.  Either way the decode
 *            lets a kernel launched after it with programmatic serialization
 *            (pa_reshape_and_cache_ex with pdl) be scheduled at once; that
 *            kernel waits for the decode before it touches memory.
 *            Engineering addition with no counterpart in the pages.
 *   early_kv nonzero (with pdl, one query per sequence, no fused append):
 *            the caller guarantees that the kernel launched just before this
 *            call writes no row of k_cache / v_cache except the newest one of
 *            each sequence (position seq_lens[s]-1), as pa_reshape_and_cache
 *            of the same step does.  The decode then starts copying the K/V
 *            rows of its first units that hold none of those positions before
 *            that kernel has finished; q, the scales and the newest rows are
 *            still read only after it.  Ignored otherwise.  A caller that
 *            breaks the guarantee gets attention over stale rows.  Engineering
 *            addition with no counterpart in the pages.
 */
typedef struct pa_decode_options {
  size_t struct_size;
  int32_t window;
  const int32_t* k_zero_point;
  const int32_t* v_zero_point;
  const void* k_new;
  const void* v_new;
  int32_t new_dtype;
  int64_t new_stride;
  const float* k_inv_scale;
  const float* v_inv_scale;
  int32_t q_len;
  int32_t pdl;
  int32_t early_kv;
} pa_decode_options;

int pa_decode_ex(void* out, pa_dtype out_dtype,
                 const void* q, pa_dtype q_dtype, int64_t q_stride,
                 const void* k_cache, const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                 const float* k_scale, const float* v_scale,
                 const int32_t* block_tables, int max_blocks_per_seq,
                 const int32_t* seq_lens,
                 int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                 float scale, int block_size, int partition_size,
                 void* workspace, size_t workspace_bytes,
                 const pa_decode_options* opt, void* stream);

/* Workspace bytes pa_decode_ex needs with these options (q_len changes the
 * size of the split records); same rules as pa_decode_workspace_bytes. */
size_t pa_decode_workspace_bytes_ex(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                    int block_size, int max_blocks_per_seq, int partition_size,
                                    pa_dtype kv_dtype, const pa_decode_options* opt);

/*
 * pa_decode_launch_config - the launch geometry pa_decode uses for these
 * sizes on the current device (introspection; nothing is launched).
 * Outputs (host pointers): resident CTAs over the device, warps per CTA,
 * K/V pipeline stages per warp and dynamic shared memory per CTA.
 */
int pa_decode_launch_config(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, int partition_size, pa_dtype q_dtype, pa_dtype kv_dtype,
                            int* ctas, int* warps_per_cta, int* stages, size_t* smem_bytes);

/*
 * pa_reshape_and_cache - write new tokens' K and V rows into their slots.
 *
 * [P2] "PagedAttention: OS仮想メモリ式の管理": blocks are handed out as tokens
 * accumulate and the block table maps token positions to physical blocks;
 * the caller encodes that mapping as one slot per token,
 *     slot = physical_block * block_size + position % block_size,
 * and this call stores k[n][h][:] at k_cache[slot/block_size][h][slot%block_size][:]
 * (v likewise) for every KV head h.  slot < 0 marks padding and is skipped.
 * 16-bit caches receive the source bits (src_dtype == kv_dtype).  FP8 caches
 * receive e4m3_rne_satfinite(float32(x) * inv_scale[h]) (product rounded in
 * float32, round-to-nearest-even, magnitudes >= 448 saturate to 448).
 *
 *   k, v           [num_tokens][num_kv_heads][head_dim] rows at k_stride /
 *                  v_stride elements per token (>= num_kv_heads*head_dim),
 *                  src_dtype F16/BF16
 *   k_cache/v_cache  pools as above (num_blocks blocks), kv_dtype
 *   slot_mapping   int64 [num_tokens]
 *   k_inv_scale/v_inv_scale  float32 [num_kv_heads]; FP8 only
 * Two tokens must not share a slot (the surviving row is then unspecified).
 */
int pa_reshape_and_cache(const void* k, const void* v, pa_dtype src_dtype,
                         int64_t k_stride, int64_t v_stride,
                         void* k_cache, void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                         const int64_t* slot_mapping, int num_tokens,
                         int num_kv_heads, int head_dim, int block_size,
                         const float* k_inv_scale, const float* v_inv_scale,
                         void* stream);

/*
 * pa_reshape_and_cache_ex - pa_reshape_and_cache with options (NULL = none).
 * opt->struct_size = sizeof(pa_cache_write_options) as compiled by the
 * caller; later fields read as 0.
 *
 *   k_zero_point / v_zero_point  int32 [num_kv_heads] device arrays in
 *            [-128, 127]; required for kv_dtype PA_INT8 ([P2] "KV量子化"),
 *            whose rows receive clamp(rne(float32(x) * inv_scale[h]) +
 *            zero_point[h], -128, 127): the product rounded in float32, then
 *            to the nearest integer with ties to even; +-inf saturate and NaN
 *            becomes +127.
 *   pdl      nonzero: launch with programmatic dependent launch.  Before
 *            it reads or writes anything, the kernel waits until the kernel
 *            launched just before it on `stream` has finished, so only the
 *            launch overlaps that kernel.  0: an ordinary launch.  Either way
 *            a decode launched after the write with pdl may start its set-up
 *            at once (it reads the cache only after the write has finished).
 *            Engineering addition with no counterpart in the pages.
 */
typedef struct pa_cache_write_options {
  size_t struct_size;
  const int32_t* k_zero_point;
  const int32_t* v_zero_point;
  int32_t pdl;
} pa_cache_write_options;

int pa_reshape_and_cache_ex(const void* k, const void* v, pa_dtype src_dtype,
                            int64_t k_stride, int64_t v_stride,
                            void* k_cache, void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                            const int64_t* slot_mapping, int num_tokens,
                            int num_kv_heads, int head_dim, int block_size,
                            const float* k_inv_scale, const float* v_inv_scale,
                            const pa_cache_write_options* opt, void* stream);

/*
 * pa_copy_blocks - the device half of copy-on-write.
 *
 * [P1] "Copy-on-Write（CoW）によるメモリ共有": before a sequence writes into a
 * block that other sequences still reference, the block manager allocates a
 * fresh block and the old block's contents are copied into it.  For every
 * pair i, physical block src_dst_pairs[2i+1] of both pools receives a copy
 * of block src_dst_pairs[2i] (all KV heads, all slots; block_bytes bytes per
 * pool, = num_kv_heads*block_size*head_dim*sizeof(element), a multiple of 16).
 * Destinations must be distinct and must not be a source of any pair (a
 * fresh block, as the pages' allocator hands out); otherwise the result is
 * unspecified.  The copy is ordered before later work on `stream`.
 *   src_dst_pairs  int32 [num_pairs][2], device
 */
int pa_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks, size_t block_bytes,
                   const int32_t* src_dst_pairs, int num_pairs, void* stream);

/*
 * pa_decode_noalloc - pa_decode for callers that cannot allocate device
 * memory (no counterpart in the pages: an engineering addition).
 *
 * A caller that runs where cudaMalloc is unavailable or forbidden at decode
 * time (an allocator-free serving loop, a process whose device memory pool
 * belongs to another framework, a plugin that is handed only its input and
 * output buffers) cannot supply pa_decode's workspace.  This entry point
 * takes the same arguments minus the workspace and uses a fixed 16 MiB
 * array that the library defines in device memory instead
 * (pa_decode_noalloc_capacity() returns its size).  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call clears the array's arrival counters on `stream`
 *     (cudaMemsetAsync) and then runs pa_decode on it.
 *   - All calls share the one array per device: calls whose kernels overlap
 *     on the GPU (different streams without ordering) race and give wrong
 *     results.  Order them on one stream or use pa_decode with workspaces.
 *   - Serves F16, BF16 and FP8 caches; an INT8 cache needs zero points,
 *     which this call has no arguments for: PA_ERR_UNSUPPORTED.
 *   - Every check of pa_decode runs before anything is enqueued; a rejected
 *     call enqueues nothing (not even the clearing of the counters).
 *   - Returns PA_ERR_WORKSPACE (detail in pa_last_error_detail) when the
 *     sizes need more split workspace than the array holds; other errors as
 *     pa_decode.
 */
int pa_decode_noalloc(void* out, pa_dtype out_dtype,
                      const void* q, pa_dtype q_dtype, int64_t q_stride,
                      const void* k_cache, const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                      const float* k_scale, const float* v_scale,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* seq_lens,
                      int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                      float scale, int block_size, int partition_size,
                      void* stream);

/* Size in bytes of the fixed device array pa_decode_noalloc uses. */
size_t pa_decode_noalloc_capacity(void);

/* Human-readable name of a pa_status value (static string). */
const char* pa_status_string(int status);

/*
 * Read and clear the current device's error word (PA_DEVERR_* bits) after
 * the work already enqueued on `stream` has finished.  Synchronises `stream`.
 * *error_bits (host pointer) receives the bits.
 */
int pa_get_device_error(void* stream, unsigned int* error_bits);

/* Text of the CUDA error behind the last PA_ERR_CUDA returned on this
 * thread ("" if none); a static thread-local string. */
const char* pa_last_error_detail(void);

/* Library ABI version (major*100 + minor). */
int pa_version(void);

/*
 * pa_debug_set_decode_wait - testing hook for the bounded waits of the decode
 * kernel (engineering addition with no counterpart in the pages; process-wide,
 * read at each later pa_decode / pa_decode_ex / pa_decode_noalloc call).
 *   limit_ns         limit of every wait of a consumer warp on its pipeline
 *                    barrier (and of the producer on a consumer's release);
 *                    0 restores the default of 2 s.  A wait that runs out
 *                    sets PA_DEVERR_TIMEOUT, the warp stops and the call's
 *                    outputs are unspecified; the kernel still returns, after
 *                    waiting (2 s at most) for its own copies in flight.
 *   withhold_copies  nonzero: the producer warp issues no copy at all, so
 *                    every consumer wait runs out (a barrier nothing
 *                    completes): the way to exercise the timeout path without
 *                    any fault.  0 for normal operation.
 * After a call that timed out, zero the workspace before its next use.
 */
void pa_debug_set_decode_wait(uint64_t limit_ns, int withhold_copies);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_PA_H */
