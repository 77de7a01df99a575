// pa_decode_static_scratch: paged decode attention for callers that cannot allocate device
// memory.  It runs the same kernels as pa_decode; only the workspace differs: here it is
// one library-owned array in device global memory, sized at compile time.
#include <cuda.h>
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
// address comes from cudaGetSymbolAddress, looked up per device (and context) below.
static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

// Address cache, one entry per device index.  An entry is valid for the CUDA context it
// was looked up in: after cudaDeviceReset the primary context is a new one and the address
// is looked up again.  A failed lookup is not cached, so a later call retries it.
struct ScratchEntry {
  CUcontext ctx = nullptr;
  void* addr = nullptr;
};
std::mutex g_mutex;
ScratchEntry g_entry[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(ptr);
    return nullptr;
  }();
  return fn;
}

CUcontext current_context() {
  CUcontext ctx = nullptr;
  const CtxGetCurrentFn fn = ctx_get_current();
  if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

// Device address of the scratch on the current device, looked up with that device current
// the first time a context is seen (cudaGetSymbolAddress allocates nothing).
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
  std::lock_guard<std::mutex> lock(g_mutex);
  ScratchEntry& ent = g_entry[dev];
  const CUcontext ctx = current_context();
  if (ctx != nullptr && ctx == ent.ctx && ent.addr != nullptr) {
    *addr = ent.addr;
    return PA_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess || p == nullptr) {
    ent = ScratchEntry{};
    char msg[200];
    snprintf(msg, sizeof msg, "pa_decode_static_scratch: scratch address lookup failed: %s",
             cudaGetErrorString(e));
    return pkv::record_error(PA_ERR_CUDA, msg);
  }
  // The lookup makes the device's primary context current if it was not yet.
  ent.ctx = ctx != nullptr ? ctx : current_context();
  ent.addr = p;
  *addr = p;
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
    // The piece counters of the in-kernel merge must start at zero.  A call leaves its own
    // counters at zero, but where they sit depends on num_seqs: after a call of another
    // size they would overlap that call's offsets or partials.  So clear them on the stream
    // first (a memset node; nothing is allocated).
    pkv::DecodePlan plan;
    if (pkv::plan_decode(num_seqs, cd.num_kv_heads, num_q_heads, max_context_len,
                         partition_tokens, &plan) == cudaSuccess &&
        plan.ws_meta_bytes > plan.ws_count_offset) {
      const cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(scratch) + plan.ws_count_offset,
                                            0, plan.ws_meta_bytes - plan.ws_count_offset,
                                            reinterpret_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof msg, "pa_decode_static_scratch: clearing the counters failed: %s",
                 cudaGetErrorString(e));
        return pkv::record_error(PA_ERR_CUDA, msg);
      }
    }
  }
  // Same argument checks, plan and kernels as pa_decode; nothing is allocated.
  return pa_decode(out, q, key_cache, value_cache, cd, block_tables, max_blocks_per_seq,
                   context_lens, num_seqs, num_q_heads, scale, max_context_len,
                   partition_tokens, scratch, num_seqs > 0 ? kScratchBytes : 0,
                   PA_LAUNCH_DEFAULT, device_status, stream);
}
