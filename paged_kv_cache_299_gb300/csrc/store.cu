// Slot mapping and KV store ("reshape_and_cache").
//
// "Tiny-vLLM" (trendpick100.com), Q&A on how Tiny-vLLM splits complexity: before the model
// runs, prepare_prefill / prepare_decode publish a slot_mapping, and a store kernel below
// the PyTorch level writes each token's key/value vector to its slot.  "vLLM"
// (blog.rlaisqls.com), section PagedAttention: slots live in 16-token blocks reached
// through a per-sequence block table.
//
// Both kernels are pure index work / data movement: the store is a bit-exact 16-byte
// vectorised copy, bound by HBM bandwidth (each token moves Hkv * D * 2 bytes of K and the
// same of V in, and the same out).
#include "common.cuh"
#include "internal.h"

namespace pkv {

// One thread per appended token.  Sequence of token t: the last s with
// query_start_loc[s] <= t (binary search; empty sequences are skipped naturally).
__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables,
                                    int32_t max_blocks_per_seq,
                                    const int32_t* __restrict__ context_lens,
                                    const int32_t* __restrict__ query_start_loc,
                                    int32_t num_seqs, int32_t num_tokens, int32_t num_blocks,
                                    int64_t* __restrict__ slot_mapping,
                                    int32_t* __restrict__ status) {
  const int32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= num_tokens) return;
  int32_t s, first, q_len;
  if (query_start_loc == nullptr) {
    s = t;
    first = t;
    q_len = 1;
  } else {
    int32_t lo = 0, hi = num_seqs - 1;
    while (lo < hi) {  // largest s in [0, num_seqs) with query_start_loc[s] <= t
      const int32_t mid = (lo + hi + 1) >> 1;
      if (query_start_loc[mid] <= t) lo = mid; else hi = mid - 1;
    }
    s = lo;
    first = query_start_loc[s];
    q_len = query_start_loc[s + 1] - first;
  }
  const int64_t pos = static_cast<int64_t>(context_lens[s]) - q_len + (t - first);
  const int64_t logical_block = pos / kBlockSize;
  if (pos < 0 || t < first || t - first >= q_len || logical_block >= max_blocks_per_seq) {
    slot_mapping[t] = -1;
    flag_error(status, PA_DEVFLAG_BAD_CONTEXT);
    return;
  }
  const int32_t phys =
      block_tables[static_cast<int64_t>(s) * max_blocks_per_seq + logical_block];
  if (phys < 0 || phys >= num_blocks) {
    slot_mapping[t] = -1;
    flag_error(status, PA_DEVFLAG_BAD_BLOCK);
    return;
  }
  slot_mapping[t] = static_cast<int64_t>(phys) * kBlockSize + pos % kBlockSize;
}

// One thread per 16-byte chunk of one token's K row (and the same chunk of its V row).
// A token's K is Hkv * 64 bf16 = Hkv * 8 chunks, read contiguously; each head's 128-byte
// row lands contiguously at cache[block][head][offset][:].
__global__ void reshape_and_cache_kernel(const uint4* __restrict__ key,
                                         const uint4* __restrict__ value,
                                         const int64_t* __restrict__ slot_mapping,
                                         int32_t num_tokens, uint4* __restrict__ key_cache,
                                         uint4* __restrict__ value_cache, int32_t num_blocks,
                                         int32_t num_kv_heads, int32_t* __restrict__ status) {
  constexpr int kChunksPerRow = kRowBytes / 16;  // 8
  const int32_t chunks_per_token = num_kv_heads * kChunksPerRow;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(num_tokens) * chunks_per_token) return;
  const int32_t t = static_cast<int32_t>(idx / chunks_per_token);
  const int32_t c = static_cast<int32_t>(idx % chunks_per_token);
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(num_blocks) * kBlockSize) {
    if (c == 0) flag_error(status, PA_DEVFLAG_BAD_SLOT);
    return;
  }
  const int32_t head = c / kChunksPerRow;
  const int32_t part = c % kChunksPerRow;
  const int64_t block = slot / kBlockSize;
  const int64_t offset = slot % kBlockSize;
  const int64_t dst = ((block * num_kv_heads + head) * kBlockSize + offset) * kChunksPerRow + part;
  const uint4 kv = ldg_nc128(key + idx);
  const uint4 vv = ldg_nc128(value + idx);
  key_cache[dst] = kv;
  value_cache[dst] = vv;
}

// Diagnostic: one warp waits on an mbarrier that nothing ever arrives on, with the same
// bounded-wait loop the pipelines use but a caller-chosen limit; when the limit passes it
// records PA_DEVFLAG_TIMEOUT and returns, leaving the context usable.
__global__ void wait_timeout_selftest_kernel(int32_t* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(&bar, 0)) {
    if (global_timer_ns() - t0 > limit_ns) {
      flag_error(status, PA_DEVFLAG_TIMEOUT);
      return;
    }
  }
}

cudaError_t launch_wait_timeout_selftest(int32_t* status, int32_t limit_ms, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(
      status, static_cast<unsigned long long>(limit_ms) * 1000000ull);
  return cudaGetLastError();
}

cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, const int32_t* query_start_loc,
                                int32_t num_seqs, int32_t num_tokens, int32_t num_blocks,
                                int64_t* slot_mapping, int32_t* status, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = (num_tokens + threads - 1) / threads;
  slot_mapping_kernel<<<blocks, threads, 0, stream>>>(block_tables, max_blocks_per_seq,
                                                      context_lens, query_start_loc, num_seqs,
                                                      num_tokens, num_blocks, slot_mapping,
                                                      status);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value,
                                     const int64_t* slot_mapping, int32_t num_tokens,
                                     void* key_cache, void* value_cache, int32_t num_blocks,
                                     int32_t num_kv_heads, int32_t* status,
                                     cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * (kRowBytes / 16);
  const int64_t blocks = (total + threads - 1) / threads;
  reshape_and_cache_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value), slot_mapping,
      num_tokens, static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), num_blocks,
      num_kv_heads, status);
  return cudaGetLastError();
}

}  // namespace pkv
