// pa_kernels.h - internal launch interface between the C ABI (pa_api.cu) and
// the kernels.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

// Default limit of every wait on a decode pipeline barrier; a wait that runs
// out records PA_DEVERR_TIMEOUT instead of hanging.  The wait for a CTA's own
// copies in flight before it exits always uses this limit.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// 8-bit caches: KV heads whose dequantisation constants the decode stages in
// shared memory (the most an 8-bit cache may have).
constexpr int kMaxHeadParams = 256;

// K/V TMA boxes are min(unit rows, block_size) whole rows; both are
// multiples of this (one 128-byte-swizzle atom is 8 x 128 bytes).
constexpr int kBoxRowQuantum = 8;

// Integer tuning override from the environment (read once per name), or -1.
int tuning_override(const char* name);

struct ReshapeArgs {
  const void* k;
  const void* v;
  int src_dtype;
  int64_t k_stride;
  int64_t v_stride;
  void* k_cache;
  void* v_cache;
  int kv_dtype;
  int64_t num_blocks;
  const int64_t* slot_mapping;
  int num_tokens;
  int num_kv_heads;
  int head_dim;
  int block_size;
  const float* k_inv_scale;
  const float* v_inv_scale;
  const int32_t* k_zero_point;  // INT8 only
  const int32_t* v_zero_point;  // INT8 only
  unsigned int* err;
  bool pdl;                     // programmatic dependent launch (the kernel waits for its predecessor first)
};

cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks, int64_t block_bytes,
                               const int32_t* pairs, int num_pairs, unsigned int* err, cudaStream_t stream);

// Everything the decode kernel reads besides the two tensor maps.
struct DecodeParams {
  void* out;
  int out_dtype;
  const void* q;
  int64_t q_stride;             // elements between consecutive sequences of q
  const float* k_scale;         // 8-bit caches only
  const float* v_scale;         // 8-bit caches only
  const int32_t* k_zero_point;  // INT8 only
  const int32_t* v_zero_point;  // INT8 only
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  int64_t num_blocks;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int group;                    // query heads per KV head (<= compiled maximum)
  float qk_scale_log2;          // softmax scale * log2(e)
  int block_size;               // tokens per cache block (a power of two >= 8)
  int block_shift;              // log2(block_size)
  int partition_units;          // 0: balanced split; >0: fixed partitions of this many units
  int frag_cost;                // balanced split: cost of a fragment besides its units, in units
  int window;                   // > 0: attend to the last `window` positions only; 0: all
  int q_len;                    // queries per sequence (their positions are the q_len newest)
  // fused append (k_new == nullptr: off): the rows of position seq_len-1
  const void* k_new;            // [num_seqs][num_kv_heads][head_dim] at new_stride elements per sequence
  const void* v_new;
  int64_t new_stride;
  int new_dtype;                // PA_F16 / PA_BF16
  const float* k_inv_scale;     // 8-bit caches: the cache write's multipliers
  const float* v_inv_scale;
  void* k_cache;                // pools, for storing the appended rows
  void* v_cache;
  float* part_records;          // split-K partial records (workspace)
  int* seg_counters;            // [num_seqs * num_kv_heads] arrival counters (workspace)
  int* pending;                 // [consumer warps][pending_cap] segments a warp merges after its loop (workspace)
  int pending_cap;
  unsigned int* err;            // per-device error word
  int stages;                   // K/V pipeline stages per warp
  int row_groups;               // consumer warps per ring (16-row variants: ceil(q_len * G / 16)); else 1
  int stage_bytes;              // bytes of one pipeline stage (several queries: K and V only)
  uint64_t wait_limit_ns;       // limit of every wait on a pipeline barrier (PA_DEVERR_TIMEOUT after it)
  int withhold_copies;          // testing hook: the producer issues no copy, so every consumer wait runs out
  int early_kv;                 // K/V of units without a sequence's newest row may be copied before the wait
};

// Compile-time variant of the decode kernel.
struct DecodeKey {
  int q_dtype;    // PA_F16 / PA_BF16
  int kv_dtype;   // PA_F16 / PA_BF16 / PA_FP8_E4M3 / PA_INT8
  int head_dim;   // 64 / 128
  int gmax;       // 1 / 4 / 8 (query heads per KV head, rounded up)
  int unit_rows;  // 16 / 32 / 64 rows per work unit
  int append;     // 1: fused append (each stage also stages the new K/V rows)
  int row_groups; // consumer warps sharing a ring (1; up to 4 for the 16-row variants)
};

// Launch geometry of one variant on the current device.
struct DecodeGeometry {
  int warps_per_cta;
  int stages;          // K/V pipeline stages per warp
  int ctas;            // resident CTAs over the whole device
  size_t smem_bytes;   // dynamic shared memory per CTA
  int record_floats;   // floats per partial record
  int stage_bytes;     // bytes of one pipeline stage
  int unit_rows;       // rows per work unit (TMA box height = min(unit_rows, block_size))
  int row_groups;      // consumer warps per ring
};

// Fills `geo` for `key` and `num_seqs` on the current device; false if the
// variant is not compiled in or the device cannot run it.
bool decode_geometry(const DecodeKey& key, int num_seqs, DecodeGeometry* geo);  // key.append selects the stage size

// Geometry and kernel attributes of the last rejected decode launch on this thread.
const char* launch_failure_note();

// pdl: launch with programmatic stream serialization, so that the kernel's
// set-up (which reads only seq_lens and block_tables) overlaps the kernel
// before it on the stream; the kernel waits for that one before anything else.
cudaError_t launch_decode(const DecodeKey& key, const DecodeGeometry& geo, const DecodeParams& p,
                          const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, cudaStream_t stream,
                          bool pdl = false);

}  // namespace pa
