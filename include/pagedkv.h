/*
 * pagedkv.h -- C ABI of libpagedkv.so, the GB300 (sm_103a) paged KV cache.
 *
 * What it computes (from the four web pages this library restates):
 *   - "vLLM" (blog.rlaisqls.com), section PagedAttention: the KV cache is cut into
 *     fixed blocks of 16 tokens; a per-sequence block table maps logical positions to
 *     physical blocks, which need not be contiguous.
 *   - "Tiny-vLLM" (trendpick100.com), Q&A on how Tiny-vLLM splits complexity:
 *     prepare_prefill / prepare_decode publish a slot_mapping, and a store kernel writes
 *     each token's key/value vector to its slot.
 *   - "vLLM", section Flash Attention: attention S = Q K^T, P = softmax(S), O = P V,
 *     evaluated block by block with a running max and running sum (online softmax), so
 *     the score matrix never reaches HBM.
 *   - "tiny-vllm (1)" (geonuchoi.com), section 2 (GQA): consecutive groups of query
 *     heads share one K/V head (query head h reads K/V head h / (Hq / Hkv)); section 1:
 *     causal decoding, position t sees positions <= t.
 *
 * Conventions shared by every call:
 *   - All pointers are DEVICE pointers on the current CUDA device, 16-byte aligned,
 *     to contiguous row-major arrays.  The caller owns every buffer; the library never
 *     allocates, frees or synchronises on these paths (pa_check_device_status aside).
 *   - bf16 tensors: key/value [T][Hkv][D], q / out [rows][Hq][D].
 *   - Cache pools: key_cache and value_cache are separate pools, each
 *     [num_blocks][Hkv][block_size][D] bf16, so one (block, kv head) tile is a
 *     contiguous block_size * D * 2 = 2 KiB run.
 *   - slot = physical_block * block_size + offset_in_block (int64); slot < 0 = skip.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Supported shapes: head_dim == 64, block_size == 16, num_q_heads / num_kv_heads in
 *     {1, 2, 4}.  Other values return PA_ERR_UNSUPPORTED.
 *
 * Errors: a call whose arguments are wrong on the host returns a negative pa_status and
 * launches nothing; pa_last_error() then holds a one-line reason.  Problems only the
 * device can see (a block id outside [0, num_blocks), a slot beyond the pool, a context
 * longer than its block-table row, a pipeline wait that timed out) never trap: the
 * kernel ORs a PA_DEVFLAG_* bit into *device_status (if non-NULL), skips the affected
 * work and returns; results of the affected rows are undefined.  Read the word with
 * pa_check_device_status().
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* same type as cudaStream_t */

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, negative size, bad desc */
  PA_ERR_UNSUPPORTED = -2,   /* a shape these kernels do not implement */
  PA_ERR_CUDA = -3,          /* a CUDA runtime call failed (launch, query, copy) */
  PA_ERR_WORKSPACE = -4,     /* workspace missing or smaller than required */
  PA_ERR_DEVICE_INDEX = -5,  /* device_status reports a bad block id / slot / length */
  PA_ERR_DEVICE_TIMEOUT = -6, /* device_status reports a pipeline wait that timed out */
  PA_ERR_OUT_OF_BLOCKS = -7   /* the block manager has too few free blocks (no change made) */
} pa_status;

/* Bits a kernel ORs into *device_status. */
#define PA_DEVFLAG_BAD_BLOCK 0x1   /* block-table entry outside [0, num_blocks) */
#define PA_DEVFLAG_BAD_SLOT 0x2    /* slot >= num_blocks * block_size */
#define PA_DEVFLAG_BAD_CONTEXT 0x4 /* context length < 0, beyond its table row, or beyond
                                      the host bound max_context_len */
#define PA_DEVFLAG_TIMEOUT 0x8     /* an mbarrier wait exceeded its time limit */
#define PA_DEVFLAG_LAYOUT 0x10     /* shared memory not aligned as the kernel requires
                                      (work skipped; reported as PA_ERR_DEVICE_INDEX) */

/* Geometry of one layer's pair of cache pools; validated on every call.  The attention
 * calls (pa_decode, pa_decode_append, pa_prefill_chunk, pa_attention_varlen) also need
 * num_blocks x num_kv_heads x 16 < 2^31 (each pool under 256 GiB): their kernels address
 * the pools as rows of 64 head dims with 32-bit coordinates; larger geometries return
 * PA_ERR_UNSUPPORTED. */
typedef struct pa_cache_desc {
  int32_t num_blocks;   /* physical blocks in each pool */
  int32_t num_kv_heads; /* Hkv (8 for Llama-3.2-1B) */
  int32_t head_dim;     /* D, must be 64 */
  int32_t block_size;   /* tokens per block, must be 16 */
} pa_cache_desc;

/* Slot mapping.  Defined by: "Tiny-vLLM" (trendpick100.com), Q&A on how Tiny-vLLM splits
 * complexity (prepare_prefill / prepare_decode publish a slot_mapping for the store), and
 * "vLLM" (blog.rlaisqls.com), section PagedAttention (16-token blocks; the block table maps
 * a logical block to its physical block).  Run here as a kernel.  Sequence s appends the
 * tokens query_start_loc[s] ..
 * query_start_loc[s+1]-1, which are the last q_len of its context_lens[s] tokens; the
 * token at logical position p gets slot block_tables[s][p / 16] * 16 + p % 16.
 *   block_tables    int32 [num_seqs][max_blocks_per_seq]
 *   context_lens    int32 [num_seqs], token count AFTER this append
 *   query_start_loc int32 [num_seqs + 1] prefix sums of appended counts, or NULL for
 *                   exactly one appended token per sequence (then num_tokens == num_seqs)
 *   num_tokens      == query_start_loc[num_seqs] (host-known; sizes the grid)
 *   slot_mapping    int64 [num_tokens] output; -1 where the device saw a bad entry
 * num_tokens == 0 is a no-op. */
pa_status pa_compute_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens,
                                  const int32_t* query_start_loc, int32_t num_seqs,
                                  int32_t num_tokens, pa_cache_desc cd,
                                  int64_t* slot_mapping, int32_t* device_status,
                                  pa_stream_t stream);

/* KV store ("reshape_and_cache").  Defined by: "Tiny-vLLM" (trendpick100.com), Q&A on how
 * Tiny-vLLM splits complexity (a store kernel writes each new token's key and value vector
 * to the slot slot_mapping names), and "vLLM", section PagedAttention (the slot lies in a
 * fixed 16-token physical block).  For every token t with slot_mapping[t] >= 0, copy
 * key[t][h][:] to key_cache[slot / 16][h][slot % 16][:] and value likewise, for all
 * heads h.  A bit-exact copy.  key/value bf16 [num_tokens][Hkv][D]; num_tokens == 0 is a
 * no-op.  Duplicate slots within one call are a caller error (the winner is undefined). */
pa_status pa_reshape_and_cache(const void* key, const void* value,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               void* key_cache, void* value_cache, pa_cache_desc cd,
                               int32_t* device_status, pa_stream_t stream);

/* Bytes of device workspace pa_decode needs for these sizes on the current device
 * (0 when the sizes are invalid).  The workspace holds the split-KV partial results, the
 * per-sequence block offsets and one piece counter per (sequence, kv head); where the
 * counters sit depends on num_seqs.  Zero-fill the buffer before its first use, and again
 * before a call whose num_seqs or num_kv_heads differ from those of the previous call on
 * it (the counters would then overlap that call's offsets or partials).  Every call whose
 * kernels run to the end leaves its counters at zero again, including calls that report a
 * device-side error through device_status (bad block id, bad context, timeout: the
 * affected pieces are still counted), so calls of the same sizes reuse the buffer without
 * clearing.  Only a CUDA error that ends a kernel early (the context is then unusable)
 * leaves the counters undefined. */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                                int32_t max_context_len, int32_t partition_tokens);

/* Launch flags of pa_decode and pa_decode_append.
 * PA_LAUNCH_OVERLAP_PREVIOUS lets the launch begin while the kernel before it in the stream
 * is still running (programmatic dependent launch), which hides the launch's start-up (the
 * block-table prefix and the first K/V tiles in flight) behind that kernel's last
 * CTAs; it carries on the launch-overhead removal of "vLLM" (blog.rlaisqls.com), section
 * CUDA Graph.  Such a launch reads block_tables, context_lens and the first K/V tiles of
 * both pools before that kernel has finished, and everything else (queries, new K/V rows,
 * outputs, workspace, device_status) only after it has finished and its writes are
 * visible.  So set it only when the kernel before it in the stream writes neither the
 * block tables nor the context lengths nor the K/V pools this call reads; the decode
 * kernels of consecutive layers of one step qualify (each layer has its own pools), a
 * store into the same pools (pa_reshape_and_cache, pa_copy_blocks, a previous
 * pa_decode_append on the same layer) does not.  The decode and chunk-prefill kernels of
 * this library (pa_prefill_chunk, pa_attention_varlen) let a following launch that carries
 * the flag start early; a launch without it waits for the previous kernel as usual.  Also
 * valid inside CUDA graph capture.
 * PA_LAUNCH_MAX_SMS(n), n in 1 .. 65535, ORed into the flags, spreads the persistent grid
 * over at most n SMs (one decode CTA or two chunk-prefill CTAs per SM) instead of all of
 * them, so that a kernel launched next with PA_LAUNCH_OVERLAP_PREVIOUS runs on the other
 * SMs at the same time: a memory-bound decode beside a tensor-core chunk prefill, as in a
 * continuous-batching step ("vLLM", section Continuous Batching).  The work is the same;
 * only where and when it runs changes, and the workspace of pa_decode_workspace_size()
 * suffices under any budget.  Other unknown bits are rejected
 * (PA_ERR_INVALID_ARG). */
#define PA_LAUNCH_DEFAULT 0u
#define PA_LAUNCH_OVERLAP_PREVIOUS 1u
#define PA_LAUNCH_MAX_SMS(n) ((uint32_t)(n) << 16)

/* Paged decode attention.  Defined by: "vLLM" (blog.rlaisqls.com), section Flash Attention
 * (S = Q K^T, P = softmax(S), O = P V, evaluated block by block with a running max and sum),
 * section PagedAttention (the K/V of a sequence are found through its block table), and
 * "tiny-vllm (1)" (geonuchoi.com), section 2 (GQA: consecutive query heads share one K/V
 * head).  One query per sequence (its newest token, already stored) over all
 * context_lens[s] cached tokens:
 *   out[s][h][:] = sum_j softmax_j(scale * q[s][h] . K_s[j][h / group]) V_s[j][h / group]
 * where K_s[j] / V_s[j] is the token at logical position j found through block_tables.
 * The (sequence, K/V head, block) tiles are split evenly over the SMs (or into runs of at
 * most partition_tokens tokens); runs that end inside a sequence leave (running max, running
 * sum, unnormalised output) partials.  With partition_tokens == 0 and max_context_len <=
 * 8192 the warp that finishes the last piece of a sequence merges them inside the same
 * kernel; otherwise a second kernel merges them.
 *   out              bf16 [num_seqs][num_q_heads][D] output
 *   q                bf16 [num_seqs][num_q_heads][D]
 *   block_tables     int32 [num_seqs][max_blocks_per_seq]
 *   context_lens     int32 [num_seqs]; 0 gives a zero output row
 *   max_context_len  host-known upper bound of context_lens (sizes the grid)
 *   partition_tokens 0 = split evenly over the device; else a multiple of 16 bounding
 *                    the run length in tokens (runs are then as even as the bound allows,
 *                    in equal numbers per streaming warp)
 *   workspace        zero-initialised device buffer of >= pa_decode_workspace_size(...)
 *                    bytes (see pa_decode_workspace_size)
 *   launch_flags     PA_LAUNCH_DEFAULT, PA_LAUNCH_OVERLAP_PREVIOUS and/or
 *                    PA_LAUNCH_MAX_SMS(n) (see there)
 * num_seqs == 0 is a no-op.  At most 4096 sequences per call. */
pa_status pa_decode(void* out, const void* q, const void* key_cache, const void* value_cache,
                    pa_cache_desc cd, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    int32_t num_seqs, int32_t num_q_heads, float scale,
                    int32_t max_context_len, int32_t partition_tokens, void* workspace,
                    size_t workspace_bytes, uint32_t launch_flags, int32_t* device_status,
                    pa_stream_t stream);

/* Decode with the store of the new tokens fused in: for every sequence s, the token at
 * position context_lens[s] - 1 (key[s][h][:], value[s][h][:], bf16 [num_seqs][Hkv][D]) is
 * written to its slot block_tables[s][(L-1) / 16] * 16 + (L-1) % 16 of both pools, and the
 * attention of pa_decode runs over all L tokens, in one launch.  Results (pools and out) are
 * bit-identical to pa_reshape_and_cache of those tokens followed by pa_decode.  This removes
 * the per-step store launches ("vLLM", CUDA Graph: per-token launch overhead; section
 * Optimized CUDA Kernels: fused kernels skip HBM round trips).  Every other argument,
 * requirement and error is that of pa_decode; a context of 0 stores nothing. */
pa_status pa_decode_append(void* out, const void* q, const void* key, const void* value,
                           void* key_cache, void* value_cache, pa_cache_desc cd,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                           float scale, int32_t max_context_len, int32_t partition_tokens,
                           void* workspace, size_t workspace_bytes, uint32_t launch_flags,
                           int32_t* device_status, pa_stream_t stream);

/* Causal chunked-prefill attention over a paged prefix.  Defined by: "tiny-vllm (1)"
 * (geonuchoi.com), section 1 (decoder-only causal attention: position t attends positions
 * <= t) and section 2 (GQA), and "vLLM" (blog.rlaisqls.com), sections Flash Attention
 * (online softmax over key blocks) and PagedAttention (paged K/V).  Sequence s has q_len =
 * query_start_loc[s+1] - query_start_loc[s] query rows, the last q_len of its
 * context_lens[s] tokens (already stored); row i sits at position L - q_len + i and
 * attends keys 0 .. L - q_len + i.  QK^T and PV run on tcgen05 tensor cores.
 *   out / q          bf16 [num_query_tokens][num_q_heads][D]
 *   num_query_tokens == query_start_loc[num_seqs], the rows of q and out (host-known;
 *                    bounds the tensor-memory-access box reads of q)
 *   max_query_len    host-known upper bound of q_len (sizes the grid; with batches beyond
 *                    2048 (sequence, 32-row tile) pairs, rows past it are not served)
 * Requires num_q_heads / num_kv_heads == 4.  num_seqs == 0 is a no-op. */
pa_status pa_prefill_chunk(void* out, const void* q, const int32_t* query_start_loc,
                           int32_t num_query_tokens, int32_t max_query_len,
                           const void* key_cache,
                           const void* value_cache, pa_cache_desc cd,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t num_seqs,
                           int32_t num_q_heads, float scale, int32_t* device_status,
                           pa_stream_t stream);

/* pa_prefill_chunk with launch flags (see PA_LAUNCH_OVERLAP_PREVIOUS and
 * PA_LAUNCH_MAX_SMS).  With PA_LAUNCH_OVERLAP_PREVIOUS the chunk kernel may run from its
 * first instruction while the previous kernel in the stream is still running (it waits for
 * that kernel only before it ends, so its completion still implies the previous kernel's):
 * set it only when that kernel writes nothing this call reads or writes (a decode of other
 * sequences without the fused store qualifies).  Results are bit-identical to
 * pa_prefill_chunk whatever the flags. */
pa_status pa_prefill_chunk_ex(void* out, const void* q, const int32_t* query_start_loc,
                              int32_t num_query_tokens, int32_t max_query_len,
                              const void* key_cache, const void* value_cache, pa_cache_desc cd,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs,
                              int32_t num_q_heads, float scale, uint32_t launch_flags,
                              int32_t* device_status, pa_stream_t stream);

/* Bytes of device workspace pa_attention_varlen needs on the current device for a batch of
 * num_seqs sequences carrying num_query_tokens query rows, for any head count and context
 * length (the decode kernel's workspace, see below; it depends on the SM count).  16 when
 * num_seqs is 0 or above 4096; 0 for negative arguments or without a device. */
size_t pa_varlen_workspace_size(int32_t num_seqs, int32_t num_query_tokens);

/* One continuous-batching step's attention ("vLLM", Continuous Batching: sequences in the
 * prefill and in the decode phase share a step).  Arguments and semantics are those of
 * pa_prefill_chunk: a sequence with q_len = 1 is a decode row, q_len > 1 a causal chunk,
 * q_len = 0 contributes nothing, and the sequences may come in any order.  Each kind runs on
 * the kernel built for it: the decode rows on the CUDA-core decode kernel of pa_decode
 * (balanced split, reading and writing their rows where query_start_loc puts them), the
 * chunks on the tensor-core kernel of pa_prefill_chunk; both launch on `stream`, and the
 * second is skipped when max_query_len is 1 (no chunk can exist).  Chunk rows are
 * bit-identical to pa_prefill_chunk; decode rows equal pa_decode's up to the rounding of its
 * split.  Batches of more than 4096 sequences run every row on the tensor-core kernel.
 *   workspace        device buffer of at least pa_varlen_workspace_size(num_seqs,
 *                    num_query_tokens) bytes, 16-byte aligned, caller-owned; no
 *                    initialisation needed: each call clears the part that must start at
 *                    zero on the stream (a memset; nothing is allocated).  Calls that can
 *                    overlap on the GPU must not share a workspace.
 * Errors: those of pa_prefill_chunk; PA_ERR_WORKSPACE for a missing, misaligned or short
 * workspace.  A query_start_loc whose rows run past num_query_tokens, or a context shorter
 * than its rows, is flagged on the device (PA_DEVFLAG_BAD_CONTEXT) and that sequence is
 * skipped. */
pa_status pa_attention_varlen(void* out, const void* q, const int32_t* query_start_loc,
                              int32_t num_query_tokens, int32_t max_query_len,
                              const void* key_cache, const void* value_cache, pa_cache_desc cd,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs,
                              int32_t num_q_heads, float scale, void* workspace,
                              size_t workspace_bytes, int32_t* device_status,
                              pa_stream_t stream);

/* pa_attention_varlen with launch flags.  PA_LAUNCH_MAX_SMS(n) (the only flag it takes)
 * puts the decode rows on n SMs and the chunks on the other SMs at the same time, instead
 * of each kernel on every SM one after the other (see PA_LAUNCH_MAX_SMS); n at or above
 * the SM count gives the default schedule.  Chunk rows are bit-identical either way;
 * decode rows may differ in their last bits (the split points of long contexts move). */
pa_status pa_attention_varlen_ex(void* out, const void* q, const int32_t* query_start_loc,
                                 int32_t num_query_tokens, int32_t max_query_len,
                                 const void* key_cache, const void* value_cache,
                                 pa_cache_desc cd, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens,
                                 int32_t num_seqs, int32_t num_q_heads, float scale,
                                 void* workspace, size_t workspace_bytes, uint32_t launch_flags,
                                 int32_t* device_status, pa_stream_t stream);

/* Paged decode attention that needs no workspace from the caller.  The vLLM and
 * tiny-vllm pages describe no counterpart for this call.  It exists for callers that cannot allocate device memory
 * themselves: code embedded in a host program that owns every device allocation (its
 * memory pool is not reachable from here), or code that must not call cudaMalloc at run
 * time because that call can stall the whole device.  It computes exactly what pa_decode
 * computes, with the same arguments minus the workspace; the split-KV partials and
 * per-sequence offsets live instead in one library-owned device array of
 * PA_DECODE_STATIC_SCRATCH_BYTES bytes, which every GPU that loads the library keeps until
 * the process exits.
 *   - Sizes whose pa_decode_workspace_size() exceeds that limit are rejected with
 *     PA_ERR_WORKSPACE before anything is launched (pa_last_error() names both sizes).
 *     Balanced splits (partition_tokens 0) need about 2.1 KB per streaming warp of the
 *     device (12 per SM) plus the offsets and counters: for up to 4096 sequences and any
 *     supported head counts they fit on GPUs of up to 280 SMs (a GB300 has 152).  Short
 *     fixed partitions over very long contexts may not fit.
 *   - The first call on a device looks up the array's device address with that device
 *     current, and again whenever the device's CUDA context has changed (for example after
 *     cudaDeviceReset); make the first call on a device before any stream capture.  A
 *     failed lookup is reported (PA_ERR_CUDA) and retried by the next call.
 *   - All calls share the array and it keeps the last call's contents.  The only part
 *     that must start at zero, the per-segment piece counters, is cleared by each call on
 *     its stream (an asynchronous memset of at most 1 MiB, before the kernels; nothing is
 *     allocated), because their place in the array depends on num_seqs; everything else
 *     is written before it is read.  Calls that can overlap on the GPU (different
 *     streams, or different host threads) race on the array: order them on one stream.
 *   - No allocation of any kind happens inside this call. */
#define PA_DECODE_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
pa_status pa_decode_static_scratch(void* out, const void* q, const void* key_cache,
                                   const void* value_cache, pa_cache_desc cd,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, float scale, int32_t max_context_len,
                                   int32_t partition_tokens, int32_t* device_status,
                                   pa_stream_t stream);

/* Copy-on-write block copy ("vLLM", PagedAttention: sequences sharing a prompt share its
 * physical blocks; a block is copied only when one of them writes into it).  For every pair
 * i, block block_mapping[2i] of both pools is copied, all heads and offsets, bit-exactly, to
 * block block_mapping[2i+1].
 *   block_mapping  int64 [num_pairs][2] (src, dst), device memory
 * Pairs must be independent: no block is both a source and a destination, no destination
 * appears twice (the order of the copies is not defined).  A pair with an id outside
 * [0, num_blocks) sets PA_DEVFLAG_BAD_BLOCK and is skipped.  num_pairs == 0 is a no-op. */
pa_status pa_copy_blocks(void* key_cache, void* value_cache, pa_cache_desc cd,
                         const int64_t* block_mapping, int32_t num_pairs,
                         int32_t* device_status, pa_stream_t stream);

/* Host-side block manager ("vLLM", PagedAttention and Continuous Batching): a pool of
 * num_blocks physical blocks of block_size tokens; each sequence owns a table of blocks,
 * grown one block at a time as tokens arrive; pa_bm_fork shares a sequence's blocks with a
 * new sequence (reference counts); appending to a sequence whose partly filled last block is
 * shared replaces that block with a fresh copy (copy-on-write) and reports the (src, dst)
 * pair for pa_copy_blocks; freeing a sequence returns the blocks no one else holds.  Not
 * thread-safe; pure host code (no CUDA calls). */
typedef struct pa_block_manager pa_block_manager;
pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, pa_block_manager** out);
void pa_bm_destroy(pa_block_manager* bm);
int32_t pa_bm_num_free_blocks(const pa_block_manager* bm);
/* Current number of sequences holding `block` (-1 for a bad id). */
int32_t pa_bm_ref_count(const pa_block_manager* bm, int32_t block);
/* New empty sequence; seq_id >= 0 and unused. */
pa_status pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id);
/* child (unused id) starts as a copy of parent: same tokens, same physical blocks. */
pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child);
/* Make room for num_tokens more tokens of seq_id.  On copy-on-write, one pair is written
 * to cow_pairs (int64 [cow_capacity][2] host array, capacity >= 1) and *num_cow = 1; copy it
 * with pa_copy_blocks before storing the new tokens.  PA_ERR_OUT_OF_BLOCKS leaves every
 * table unchanged. */
pa_status pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, int32_t num_tokens,
                              int64_t* cow_pairs, int32_t cow_capacity, int32_t* num_cow);
pa_status pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id);
/* Tokens held by seq_id (-1 if unknown). */
int64_t pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq_id);
/* Writes seq_id's physical block ids to out[0..n) and -1 to out[n..max_blocks); returns n,
 * or a negative pa_status when the sequence is unknown or has more than max_blocks blocks. */
int32_t pa_bm_block_table(const pa_block_manager* bm, int64_t seq_id, int32_t* out,
                          int32_t max_blocks);

/* Diagnostic for the failure path: launches one warp that waits on an mbarrier nothing
 * arrives on, using the bounded wait of the pipelines with a limit of limit_ms (1..1000);
 * when it expires the kernel sets PA_DEVFLAG_TIMEOUT in *device_status and returns.  Lets a
 * test confirm that a stalled pipeline reports instead of hanging and leaves the context
 * usable.  No counterpart on the pages (engineering support only). */
pa_status pa_selftest_wait_timeout(int32_t* device_status, int32_t limit_ms,
                                   pa_stream_t stream);

/* Measurement support: read `bytes` (a multiple of 16) of device memory at `buf` once with
 * 16-byte streaming loads, in one kernel launch, and XOR all its 32-bit words into
 * *xor_out (a device uint32; zero it first to obtain the XOR of the buffer), so the reads
 * cannot be skipped and the result can be checked.  It is the in-run read-only reference
 * against which the decode kernel's KV bandwidth is reported (same bytes, same launch
 * conditions).  bytes == 0 launches nothing (buf may then be NULL).  No counterpart on the
 * pages. */
pa_status pa_stream_read(const void* buf, size_t bytes, uint32_t* xor_out, pa_stream_t stream);

/* Synchronise `stream`, read *device_status and translate it: PA_OK when zero,
 * PA_ERR_DEVICE_TIMEOUT when the timeout bit is set, else PA_ERR_DEVICE_INDEX. */
pa_status pa_check_device_status(const int32_t* device_status, pa_stream_t stream);

/* Static description of a status code (never NULL). */
const char* pa_status_string(pa_status status);

/* One-line detail of this thread's last non-OK return ("" if none). */
const char* pa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
