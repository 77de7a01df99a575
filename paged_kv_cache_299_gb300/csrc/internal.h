// Host-side launchers shared between the C-ABI entry points (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, const int32_t* query_start_loc,
                                int32_t num_seqs, int32_t num_tokens, int32_t num_blocks,
                                int64_t* slot_mapping, int32_t* status, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const void* key, const void* value,
                                     const int64_t* slot_mapping, int32_t num_tokens,
                                     void* key_cache, void* value_cache, int32_t num_blocks,
                                     int32_t num_kv_heads, int32_t* status,
                                     cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(int32_t* status, int32_t limit_ms, cudaStream_t stream);
cudaError_t launch_stream_read(const void* buf, size_t bytes, uint32_t* x, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* key_cache, void* value_cache, const int64_t* block_mapping,
                               int32_t num_pairs, int32_t num_blocks, int32_t num_kv_heads,
                               int32_t* status, cudaStream_t stream);

// Work decomposition of one pa_decode call (identical in the size query and the call).
struct DecodePlan {
  int group;          // q heads per kv head
  int grid;           // CTAs of the attention kernel (persistent, <= resident capacity)
  int runs;           // units of the tile decomposition; CTA c serves runs c, c + grid, ...
  int chunk;          // tiles per run (fixed mode), 0 = balanced split of the real total
  int64_t tile_bound; // > 0: host upper bound of the tile count, checked on the device
  size_t smem_bytes;  // dynamic shared memory of the attention kernel
  bool fused_merge;          // split segments merged inside the attention kernel
  bool merge_split_heads;    // otherwise: the merge kernel takes one CTA per query head
  bool prefetch_ok;          // warps may ask L2 for tiles past their ring before the wait
  size_t ws_count_offset;    // offset of the per-segment piece counters (must start zeroed)
  size_t ws_meta_bytes;      // offset of the partials inside the workspace
  size_t workspace_bytes;    // total workspace
};

// Returns cudaSuccess and fills `plan`, or an error (e.g. no device).
// max_sms > 0 confines the persistent grid to that many SMs (the rest stay free for a
// kernel launched beside it).
cudaError_t plan_decode(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                        int32_t max_context_len, int32_t partition_tokens, DecodePlan* plan,
                        int32_t max_sms = 0);

struct DecodeArgs {
  void* out;
  const void* q;
  const void* key_cache;
  const void* value_cache;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t num_blocks;
  float scale;
  void* workspace;
  int32_t* status;
  const void* k_new = nullptr;  // fused append (pa_decode_append), else null
  const void* v_new = nullptr;
  const int32_t* q_rows = nullptr;  // mixed batch: query/output row per sequence (prefix sums
                                    // of q_len); only q_len == 1 sequences are served
  int32_t num_query_tokens = 0;
  // Programmatic dependent launch: the kernel may start before the previous kernel in the
  // stream has finished; it reads block_tables, context_lens (and q_rows) and its first
  // K/V tiles before waiting for that kernel, everything else after.
  bool overlap_previous = false;
};

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);

// Tensor map of a [rows][64] bf16 array read in boxes of `box_rows` rows with the 128-byte
// swizzle (the K/V pools, rows = blocks x kv heads x 16); false if the driver call fails.
bool encode_pool_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);

struct PrefillArgs {
  void* out;
  const void* q;
  const int32_t* query_start_loc;
  int32_t num_query_tokens;
  int32_t max_query_len;
  const void* key_cache;
  const void* value_cache;
  int32_t num_blocks;
  int32_t num_kv_heads;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;
  int32_t num_seqs;
  int32_t num_q_heads;
  float scale;
  int32_t* status;
};

// overlap_previous: programmatic dependent launch behind the previous kernel in the stream
// (the kernel waits for it only at its end); max_sms > 0: at most two CTAs on each of that
// many SMs.
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream, bool overlap_previous = false,
                           int32_t max_sms = 0);

// Unified varlen launch: the decode kernel serves the one-row sequences in place (the
// workspace is its workspace), the chunk kernel the others.  Sizes on the current device:
// an upper bound for any head count and context (the size query), and the exact need of
// one call.
int decode_max_seqs();
size_t varlen_workspace_size(int32_t num_seqs, int32_t num_query_tokens);
size_t varlen_workspace_need(const PrefillArgs& a);
// decode_sms in 1 .. SMs-1: the decode rows on that many SMs and the chunks on the others,
// at the same time; 0: each kernel on every SM, one after the other.
cudaError_t launch_varlen(const PrefillArgs& a, void* workspace, cudaStream_t stream,
                          int32_t decode_sms = 0);

}  // namespace pkv
