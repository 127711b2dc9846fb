// Internal interface between the decode launcher (paged_attn_decode.cu) and the
// kernel for partitions that several sequences share (paged_attn_shared.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pagedkv {

struct SharedParams {
  const void* q;             // [N][H][D]
  const void* k_cache;       // [B][H][bs][D]
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* records;    // [num_records][PA_SHARE_RECORD_WORDS]
  const int32_t* tail_start; // [N] or null: where a member's own part of a prefix
                             // record's partition begins
  const int32_t* record_count;  // optional: the records to run (num_records: capacity)
  int num_records;
  int num_seqs;
  int num_heads;
  int block_size;
  int max_blocks;
  int num_blocks;
  int partition_tokens;
  int num_partitions;        // P of the workspace layout
  int heads_per_cta;         // G
  int stages;                // S
  int fused_append;          // lengths include a token appended by this step
  int out_dtype;
  float qscale;              // scale * log2(e)
  void* out;                 // [N][H][D], for members whose only partition is shared
  float* ws_acc;
  float2* ws_ml;
  int32_t* err;
};

// Shared memory of one block of the shared-partition kernel.
size_t shared_kernel_smem_bytes(int head_dim, int heads_per_cta, int stages);

// Enqueue the kernel over all records; returns a pa_status.  Its blocks trigger
// programmatic dependents when they start (the per-sequence partition pass is
// launched after it as one).
int launch_shared_partitions(const SharedParams& p, int dtype, int head_dim, cudaStream_t stream);

}  // namespace pagedkv
