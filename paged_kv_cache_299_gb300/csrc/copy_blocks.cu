// Block copy for copy-on-write ("vLLM", blog.rlaisqls.com, section PagedAttention: requests
// that share a prompt (beam search, parallel sampling) share its physical blocks, and a block
// is copied only when one of them writes into it).
//
// Pure data movement, HBM-bound: every pair moves one whole block of both pools
// (Hkv x 16 x 64 bf16 = 16 KiB each for 8 kv heads).  One thread per 16-byte chunk; the
// chunks of one block are contiguous, so reads and writes are fully coalesced.
#include "common.cuh"
#include "internal.h"

namespace pkv {

__global__ void copy_blocks_kernel(uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                                   const int64_t* __restrict__ block_mapping, int32_t num_pairs,
                                   int32_t num_blocks, int32_t chunks_per_block,
                                   int32_t* __restrict__ status) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(num_pairs) * chunks_per_block) return;
  const int32_t pair = static_cast<int32_t>(idx / chunks_per_block);
  const int32_t c = static_cast<int32_t>(idx % chunks_per_block);
  const int64_t src = block_mapping[2 * pair];
  const int64_t dst = block_mapping[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (c == 0) flag_error(status, PA_DEVFLAG_BAD_BLOCK);
    return;
  }
  const int64_t from = src * chunks_per_block + c;
  const int64_t to = dst * chunks_per_block + c;
  const uint4 k = ldg_nc128(key_cache + from);
  const uint4 v = ldg_nc128(value_cache + from);
  key_cache[to] = k;
  value_cache[to] = v;
}

cudaError_t launch_copy_blocks(void* key_cache, void* value_cache, const int64_t* block_mapping,
                               int32_t num_pairs, int32_t num_blocks, int32_t num_kv_heads,
                               int32_t* status, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int32_t chunks = num_kv_heads * kTileBytes / 16;
  const int threads = 256;
  const int64_t total = static_cast<int64_t>(num_pairs) * chunks;
  copy_blocks_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, stream>>>(
      static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), block_mapping, num_pairs,
      num_blocks, chunks, status);
  return cudaGetLastError();
}

}  // namespace pkv
