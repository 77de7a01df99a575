// C-ABI entry points of libpagedkv.so: host-side argument checks, then kernel launches.
// Declarations and the contract of every call are in include/pagedkv.h.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
int decode_max_seqs();
}  // namespace pkv

namespace {

// the launch-flag bits the attention calls accept (the SM budget takes bits 16-31)
constexpr uint32_t kKnownLaunchFlags = PA_LAUNCH_OVERLAP_PREVIOUS | 0xFFFF0000u;

thread_local char g_last_error[256] = "";

pa_status fail(pa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

pa_status ok() {
  g_last_error[0] = '\0';
  return PA_OK;
}

pa_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status check_desc(const pa_cache_desc& cd) {
  if (cd.num_blocks <= 0 || cd.num_kv_heads <= 0 || cd.num_kv_heads > 64)
    return fail(PA_ERR_INVALID_ARG, "cache desc: num_blocks %d, num_kv_heads %d",
                cd.num_blocks, cd.num_kv_heads);
  if (cd.head_dim != pkv::kHeadDim)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d (only 64 is implemented)", cd.head_dim);
  if (cd.block_size != pkv::kBlockSize)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (only 16 is implemented)", cd.block_size);
  return PA_OK;
}

// The attention kernels read the pools through tensor maps over [blocks x heads x 16][64]
// rows with 32-bit row coordinates: fewer than 2^31 rows (each pool under 256 GiB).
pa_status check_attention_pools(const pa_cache_desc& cd) {
  pa_status st = check_desc(cd);
  if (st != PA_OK) return st;
  const int64_t rows = static_cast<int64_t>(cd.num_blocks) * cd.num_kv_heads * cd.block_size;
  if (rows >= (int64_t{1} << 31))
    return fail(PA_ERR_UNSUPPORTED,
                "cache desc: %d blocks x %d kv heads x 16 rows = %lld rows per pool (the "
                "attention kernels take fewer than 2^31)",
                cd.num_blocks, cd.num_kv_heads, static_cast<long long>(rows));
  return PA_OK;
}

}  // namespace

namespace pkv {
// Lets other translation units of the library report a host-side rejection through
// pa_last_error().
pa_status record_error(pa_status st, const char* message) {
  return fail(st, "%s", message);
}
}  // namespace pkv

extern "C" {

pa_status pa_compute_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens,
                                  const int32_t* query_start_loc, int32_t num_seqs,
                                  int32_t num_tokens, pa_cache_desc cd,
                                  int64_t* slot_mapping, int32_t* device_status,
                                  pa_stream_t stream) {
  pa_status st = check_desc(cd);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_tokens %d, num_seqs %d, max_blocks_per_seq %d",
                num_tokens, num_seqs, max_blocks_per_seq);
  if (num_tokens == 0) return ok();
  if (num_seqs == 0) return fail(PA_ERR_INVALID_ARG, "tokens without sequences");
  if (query_start_loc == nullptr && num_tokens != num_seqs)
    return fail(PA_ERR_INVALID_ARG, "query_start_loc NULL needs num_tokens == num_seqs");
  if (!block_tables || !context_lens || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  return from_cuda(pkv::launch_slot_mapping(block_tables, max_blocks_per_seq, context_lens,
                                            query_start_loc, num_seqs, num_tokens,
                                            cd.num_blocks, slot_mapping, device_status,
                                            reinterpret_cast<cudaStream_t>(stream)),
                   "slot mapping launch");
}

pa_status pa_reshape_and_cache(const void* key, const void* value,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               void* key_cache, void* value_cache, pa_cache_desc cd,
                               int32_t* device_status, pa_stream_t stream) {
  pa_status st = check_desc(cd);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
  if (num_tokens == 0) return ok();
  if (!key || !value || !slot_mapping || !key_cache || !value_cache)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PA_ERR_INVALID_ARG, "key/value/cache pointers must be 16-byte aligned");
  return from_cuda(pkv::launch_reshape_and_cache(key, value, slot_mapping, num_tokens,
                                                 key_cache, value_cache, cd.num_blocks,
                                                 cd.num_kv_heads, device_status,
                                                 reinterpret_cast<cudaStream_t>(stream)),
                   "reshape_and_cache launch");
}

static pa_status check_decode_sizes(int32_t num_seqs, int32_t num_kv_heads,
                                    int32_t num_q_heads, int32_t max_context_len,
                                    int32_t partition_tokens) {
  if (num_seqs < 0 || num_seqs > pkv::decode_max_seqs())
    return fail(num_seqs < 0 ? PA_ERR_INVALID_ARG : PA_ERR_UNSUPPORTED,
                "num_seqs %d (0..%d supported)", num_seqs, pkv::decode_max_seqs());
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d",
                num_q_heads, num_kv_heads);
  const int group = num_q_heads / num_kv_heads;
  if (group != 1 && group != 2 && group != 4)
    return fail(PA_ERR_UNSUPPORTED, "query heads per kv head %d (1, 2, 4 implemented)", group);
  if (max_context_len < 0) return fail(PA_ERR_INVALID_ARG, "max_context_len %d", max_context_len);
  if (partition_tokens < 0 || partition_tokens % pkv::kBlockSize != 0)
    return fail(PA_ERR_INVALID_ARG, "partition_tokens %d (0 or a multiple of 16)",
                partition_tokens);
  return PA_OK;
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                                int32_t max_context_len, int32_t partition_tokens) {
  if (check_decode_sizes(num_seqs, num_kv_heads, num_q_heads, max_context_len,
                         partition_tokens) != PA_OK)
    return 0;
  if (num_seqs == 0) return 0;
  pkv::DecodePlan plan;
  if (pkv::plan_decode(num_seqs, num_kv_heads, num_q_heads, max_context_len, partition_tokens,
                       &plan) != cudaSuccess)
    return 0;
  return plan.workspace_bytes;
}

static pa_status decode_impl(void* out, const void* q, const void* k_new, const void* v_new,
                             const void* key_cache, const void* value_cache,
                    pa_cache_desc cd, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    int32_t num_seqs, int32_t num_q_heads, float scale,
                    int32_t max_context_len, int32_t partition_tokens, void* workspace,
                    size_t workspace_bytes, uint32_t launch_flags, int32_t* device_status,
                    pa_stream_t stream) {
  pa_status st = check_attention_pools(cd);
  if (st != PA_OK) return st;
  st = check_decode_sizes(num_seqs, cd.num_kv_heads, num_q_heads, max_context_len,
                          partition_tokens);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return ok();
  if (max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq %d", max_blocks_per_seq);
  if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PA_ERR_INVALID_ARG, "out/q/cache pointers must be 16-byte aligned");
  if (!(scale > 0.f) || !isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale %g", scale);
  if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
    return fail(PA_ERR_INVALID_ARG, "k_new / v_new: both or neither, 16-byte aligned");
  if (launch_flags & ~kKnownLaunchFlags)
    return fail(PA_ERR_INVALID_ARG, "unknown launch flags 0x%x", launch_flags);
  pkv::DecodePlan plan;
  cudaError_t e = pkv::plan_decode(num_seqs, cd.num_kv_heads, num_q_heads, max_context_len,
                                   partition_tokens, &plan, static_cast<int32_t>(launch_flags >> 16));
  if (e != cudaSuccess) return from_cuda(e, "decode plan");
  if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned16(workspace))
    return fail(PA_ERR_WORKSPACE, "workspace %zu bytes at %p, need %zu (16-byte aligned)",
                workspace_bytes, workspace, plan.workspace_bytes);
  pkv::DecodeArgs a;
  a.out = out;
  a.q = q;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = cd.num_kv_heads;
  a.num_blocks = cd.num_blocks;
  a.scale = scale;
  a.workspace = workspace;
  a.status = device_status;
  a.k_new = k_new;
  a.v_new = v_new;
  a.overlap_previous = (launch_flags & PA_LAUNCH_OVERLAP_PREVIOUS) != 0;
  return from_cuda(pkv::launch_decode(a, plan, reinterpret_cast<cudaStream_t>(stream)),
                   "decode launch");
}

pa_status pa_decode(void* out, const void* q, const void* key_cache, const void* value_cache,
                    pa_cache_desc cd, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    int32_t num_seqs, int32_t num_q_heads, float scale,
                    int32_t max_context_len, int32_t partition_tokens, void* workspace,
                    size_t workspace_bytes, uint32_t launch_flags, int32_t* device_status,
                    pa_stream_t stream) {
  return decode_impl(out, q, nullptr, nullptr, key_cache, value_cache, cd, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, num_q_heads, scale,
                     max_context_len, partition_tokens, workspace, workspace_bytes,
                     launch_flags, device_status, stream);
}

pa_status pa_decode_append(void* out, const void* q, const void* key, const void* value,
                           void* key_cache, void* value_cache, pa_cache_desc cd,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                           float scale, int32_t max_context_len, int32_t partition_tokens,
                           void* workspace, size_t workspace_bytes, uint32_t launch_flags,
                           int32_t* device_status, pa_stream_t stream) {
  if (num_seqs > 0 && (!key || !value)) return fail(PA_ERR_INVALID_ARG, "null key/value");
  return decode_impl(out, q, key, value, key_cache, value_cache, cd, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, num_q_heads, scale,
                     max_context_len, partition_tokens, workspace, workspace_bytes,
                     launch_flags, device_status, stream);
}

namespace {

// Validation and argument packing shared by pa_prefill_chunk and pa_attention_varlen;
// returns PA_OK with *skip set when there is nothing to do.
pa_status chunk_args(void* out, const void* q, const int32_t* query_start_loc,
                     int32_t num_query_tokens, int32_t max_query_len, const void* key_cache,
                     const void* value_cache, pa_cache_desc cd, const int32_t* block_tables,
                     int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                     int32_t num_q_heads, float scale, int32_t* device_status,
                     pkv::PrefillArgs* a, bool* skip) {
  *skip = false;
  pa_status st = check_attention_pools(cd);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || max_query_len < 0 || num_query_tokens < 0 || max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG,
                "num_seqs %d, num_query_tokens %d, max_query_len %d, max_blocks_per_seq %d",
                num_seqs, num_query_tokens, max_query_len, max_blocks_per_seq);
  if (num_seqs == 0 || max_query_len == 0 || num_query_tokens == 0) {
    *skip = true;
    return PA_OK;
  }
  if (max_query_len > num_query_tokens)
    return fail(PA_ERR_INVALID_ARG, "max_query_len %d > num_query_tokens %d", max_query_len,
                num_query_tokens);
  if (num_q_heads != 4 * cd.num_kv_heads)
    return fail(PA_ERR_UNSUPPORTED, "prefill needs 4 query heads per kv head (got %d / %d)",
                num_q_heads, cd.num_kv_heads);
  if (!out || !q || !query_start_loc || !key_cache || !value_cache || !block_tables ||
      !context_lens)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PA_ERR_INVALID_ARG, "out/q/cache pointers must be 16-byte aligned");
  if (!(scale > 0.f) || !isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale %g", scale);
  a->out = out;
  a->q = q;
  a->query_start_loc = query_start_loc;
  a->num_query_tokens = num_query_tokens;
  a->max_query_len = max_query_len;
  a->key_cache = key_cache;
  a->value_cache = value_cache;
  a->num_blocks = cd.num_blocks;
  a->num_kv_heads = cd.num_kv_heads;
  a->block_tables = block_tables;
  a->max_blocks_per_seq = max_blocks_per_seq;
  a->context_lens = context_lens;
  a->num_seqs = num_seqs;
  a->num_q_heads = num_q_heads;
  a->scale = scale;
  a->status = device_status;
  return PA_OK;
}

}  // namespace

pa_status pa_prefill_chunk_ex(void* out, const void* q, const int32_t* query_start_loc,
                              int32_t num_query_tokens, int32_t max_query_len,
                              const void* key_cache, const void* value_cache, pa_cache_desc cd,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs,
                              int32_t num_q_heads, float scale, uint32_t launch_flags,
                              int32_t* device_status, pa_stream_t stream) {
  pkv::PrefillArgs a;
  bool skip;
  pa_status st = chunk_args(out, q, query_start_loc, num_query_tokens, max_query_len, key_cache,
                            value_cache, cd, block_tables, max_blocks_per_seq, context_lens,
                            num_seqs, num_q_heads, scale, device_status, &a, &skip);
  if (st != PA_OK) return st;
  if (launch_flags & ~kKnownLaunchFlags)
    return fail(PA_ERR_INVALID_ARG, "unknown launch flags 0x%x", launch_flags);
  if (skip) return ok();
  return from_cuda(pkv::launch_prefill(a, reinterpret_cast<cudaStream_t>(stream),
                                       (launch_flags & PA_LAUNCH_OVERLAP_PREVIOUS) != 0,
                                       static_cast<int32_t>(launch_flags >> 16)),
                   "prefill launch");
}

pa_status pa_prefill_chunk(void* out, const void* q, const int32_t* query_start_loc,
                           int32_t num_query_tokens, int32_t max_query_len,
                           const void* key_cache,
                           const void* value_cache, pa_cache_desc cd,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t num_seqs,
                           int32_t num_q_heads, float scale, int32_t* device_status,
                           pa_stream_t stream) {
  return pa_prefill_chunk_ex(out, q, query_start_loc, num_query_tokens, max_query_len,
                             key_cache, value_cache, cd, block_tables, max_blocks_per_seq,
                             context_lens, num_seqs, num_q_heads, scale, PA_LAUNCH_DEFAULT,
                             device_status, stream);
}

size_t pa_varlen_workspace_size(int32_t num_seqs, int32_t num_query_tokens) {
  if (num_seqs < 0 || num_query_tokens < 0) return 0;
  if (num_seqs == 0) return 16;
  return pkv::varlen_workspace_size(num_seqs, num_query_tokens);
}

pa_status pa_attention_varlen_ex(void* out, const void* q, const int32_t* query_start_loc,
                                 int32_t num_query_tokens, int32_t max_query_len,
                                 const void* key_cache, const void* value_cache,
                                 pa_cache_desc cd, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens,
                                 int32_t num_seqs, int32_t num_q_heads, float scale,
                                 void* workspace, size_t workspace_bytes, uint32_t launch_flags,
                                 int32_t* device_status, pa_stream_t stream) {
  pkv::PrefillArgs a;
  bool skip;
  pa_status st = chunk_args(out, q, query_start_loc, num_query_tokens, max_query_len, key_cache,
                            value_cache, cd, block_tables, max_blocks_per_seq, context_lens,
                            num_seqs, num_q_heads, scale, device_status, &a, &skip);
  if (st != PA_OK) return st;
  if (launch_flags & ~0xFFFF0000u)  // only the decode rows' SM budget
    return fail(PA_ERR_INVALID_ARG, "unknown launch flags 0x%x", launch_flags);
  if (skip) return ok();
  if (!workspace || !aligned16(workspace))
    return fail(PA_ERR_WORKSPACE, "varlen workspace at %p (needs a 16-byte aligned buffer)",
                workspace);
  const size_t need = pkv::varlen_workspace_need(a);
  if (need == 0) return fail(PA_ERR_CUDA, "varlen: decode plan failed (no device?)");
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE, "varlen workspace %zu bytes, need %zu", workspace_bytes, need);
  return from_cuda(pkv::launch_varlen(a, workspace, reinterpret_cast<cudaStream_t>(stream),
                                      static_cast<int32_t>(launch_flags >> 16)),
                   "varlen launch");
}

pa_status pa_attention_varlen(void* out, const void* q, const int32_t* query_start_loc,
                              int32_t num_query_tokens, int32_t max_query_len,
                              const void* key_cache, const void* value_cache, pa_cache_desc cd,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs,
                              int32_t num_q_heads, float scale, void* workspace,
                              size_t workspace_bytes, int32_t* device_status,
                              pa_stream_t stream) {
  return pa_attention_varlen_ex(out, q, query_start_loc, num_query_tokens, max_query_len,
                                key_cache, value_cache, cd, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_q_heads, scale, workspace,
                                workspace_bytes, PA_LAUNCH_DEFAULT, device_status, stream);
}

pa_status pa_copy_blocks(void* key_cache, void* value_cache, pa_cache_desc cd,
                         const int64_t* block_mapping, int32_t num_pairs,
                         int32_t* device_status, pa_stream_t stream) {
  pa_status st = check_desc(cd);
  if (st != PA_OK) return st;
  if (num_pairs < 0) return fail(PA_ERR_INVALID_ARG, "num_pairs %d", num_pairs);
  if (num_pairs == 0) return ok();
  if (!key_cache || !value_cache || !block_mapping) return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(key_cache) || !aligned16(value_cache))
    return fail(PA_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  return from_cuda(pkv::launch_copy_blocks(key_cache, value_cache, block_mapping, num_pairs,
                                           cd.num_blocks, cd.num_kv_heads, device_status,
                                           reinterpret_cast<cudaStream_t>(stream)),
                   "copy_blocks launch");
}

pa_status pa_selftest_wait_timeout(int32_t* device_status, int32_t limit_ms,
                                   pa_stream_t stream) {
  if (!device_status) return fail(PA_ERR_INVALID_ARG, "null status pointer");
  if (limit_ms < 1 || limit_ms > 1000) return fail(PA_ERR_INVALID_ARG, "limit_ms %d", limit_ms);
  return from_cuda(pkv::launch_wait_timeout_selftest(device_status, limit_ms,
                                                     reinterpret_cast<cudaStream_t>(stream)),
                   "timeout self-test launch");
}

pa_status pa_stream_read(const void* buf, size_t bytes, uint32_t* xor_out, pa_stream_t stream) {
  if (!xor_out || (reinterpret_cast<uintptr_t>(xor_out) & 3u) != 0)
    return fail(PA_ERR_INVALID_ARG, "null or misaligned xor_out");
  if (bytes % 16 != 0) return fail(PA_ERR_INVALID_ARG, "bytes %zu not a multiple of 16", bytes);
  if (bytes > 0 && (!buf || !aligned16(buf)))
    return fail(PA_ERR_INVALID_ARG, "null or misaligned buffer");
  return from_cuda(pkv::launch_stream_read(buf, bytes, xor_out, reinterpret_cast<cudaStream_t>(stream)),
                   "stream read launch");
}

pa_status pa_check_device_status(const int32_t* device_status, pa_stream_t stream) {
  if (!device_status) return fail(PA_ERR_INVALID_ARG, "null status pointer");
  int32_t word = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&word, device_status, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return from_cuda(e, "reading device status");
  if (word == 0) return ok();
  if (word & PA_DEVFLAG_TIMEOUT)
    return fail(PA_ERR_DEVICE_TIMEOUT, "device status 0x%x: a pipeline wait timed out", word);
  return fail(PA_ERR_DEVICE_INDEX, "device status 0x%x:%s%s%s", word,
              (word & PA_DEVFLAG_BAD_BLOCK) ? " bad block id" : "",
              (word & PA_DEVFLAG_BAD_SLOT) ? " slot beyond pool" : "",
              (word & PA_DEVFLAG_BAD_CONTEXT) ? " bad context length" : "");
}

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_DEVICE_INDEX: return "device reported a bad index";
    case PA_ERR_DEVICE_TIMEOUT: return "device reported a wait timeout";
    case PA_ERR_OUT_OF_BLOCKS: return "not enough free blocks";
  }
  return "unknown status";
}

const char* pa_last_error(void) { return g_last_error; }

}  // extern "C"
