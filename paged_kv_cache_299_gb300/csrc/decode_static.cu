// pa_decode_static_scratch: paged decode attention for callers that cannot allocate device
// memory.  It runs the same kernels as pa_decode; only the workspace differs: here it is
// one library-owned array in device global memory, sized at compile time.
#include <mutex>
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
pa_status record_error(pa_status st, const char* message);
}  // namespace pkv

namespace {

constexpr size_t kScratchBytes = PA_DECODE_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name only stands in for the array: its device
// address comes from cudaGetSymbolAddress, looked up once per device below.
static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

std::once_flag g_setup_once[kMaxDevices];
void* g_scratch_addr[kMaxDevices] = {};
cudaError_t g_setup_status[kMaxDevices] = {};

// Device address of the scratch on the current device (set up on first use).
pa_status scratch_on_current_device(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    return pkv::record_error(PA_ERR_CUDA, "pa_decode_static_scratch: no current CUDA device");
  }
  if (dev < 0 || dev >= kMaxDevices) {
    return pkv::record_error(PA_ERR_UNSUPPORTED,
                             "pa_decode_static_scratch: device index beyond 63");
  }
  std::call_once(g_setup_once[dev], [dev]() {
    void* p = nullptr;
    g_setup_status[dev] = cudaGetSymbolAddress(&p, g_decode_scratch);
    g_scratch_addr[dev] = p;
  });
  if (g_setup_status[dev] != cudaSuccess || g_scratch_addr[dev] == nullptr) {
    char msg[200];
    snprintf(msg, sizeof msg, "pa_decode_static_scratch: scratch address lookup failed: %s",
             cudaGetErrorString(g_setup_status[dev]));
    return pkv::record_error(PA_ERR_CUDA, msg);
  }
  *addr = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_static_scratch(
    void* out, const void* q, const void* key_cache, const void* value_cache, pa_cache_desc cd,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t num_seqs, int32_t num_q_heads, float scale, int32_t max_context_len,
    int32_t partition_tokens, int32_t* device_status, pa_stream_t stream) {
  if (num_seqs > 0) {
    const size_t need = pa_decode_workspace_size(num_seqs, cd.num_kv_heads, num_q_heads,
                                                 max_context_len, partition_tokens);
    if (need > kScratchBytes) {
      char msg[200];
      snprintf(msg, sizeof msg,
               "pa_decode_static_scratch: these sizes need %zu bytes of workspace, the "
               "built-in scratch holds %zu; call pa_decode with a workspace instead",
               need, kScratchBytes);
      return pkv::record_error(PA_ERR_WORKSPACE, msg);
    }
  }
  void* scratch = nullptr;
  if (num_seqs > 0) {
    const pa_status st = scratch_on_current_device(&scratch);
    if (st != PA_OK) return st;
  }
  // Same argument checks, plan and kernels as pa_decode; nothing is allocated.
  return pa_decode(out, q, key_cache, value_cache, cd, block_tables, max_blocks_per_seq,
                   context_lens, num_seqs, num_q_heads, scale, max_context_len,
                   partition_tokens, scratch, num_seqs > 0 ? kScratchBytes : 0,
                   device_status, stream);
}
