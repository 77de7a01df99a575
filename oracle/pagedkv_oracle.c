/*
 * Paged KV-cache oracle: a plain, slow, single-threaded CPU restatement of what the
 * paged KV-cache hot path computes.  TEST INFRASTRUCTURE ONLY: the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load it; the product library never
 * does, and this file shares no code, header or table with the CUDA path.
 *
 * Sources (the four web pages this project restates):
 *   - "vLLM" (blog.rlaisqls.com), section PagedAttention, "virtual-memory style":
 *     the KV cache is cut into fixed blocks of 16 tokens; a per-sequence table maps
 *     logical positions to physical blocks, which need not be contiguous; 300 tokens
 *     use 19 blocks and waste the last block's 4 free slots.
 *   - "Tiny-vLLM" (trendpick100.com), Q&A on how Tiny-vLLM splits complexity:
 *     prepare_prefill / prepare_decode publish a slot_mapping that tells the store
 *     kernel where each token's key/value vector is written.
 *   - "tiny-vllm (1)" (geonuchoi.com), section 2 (GQA) figure: query heads 0-3 share
 *     K/V head 0, query heads 4.. share K/V head 1, ...; section 1: causal decoding,
 *     token t sees tokens 1..t only.
 *   - "vLLM", section Flash Attention: standard attention S = Q K^T, P = softmax(S),
 *     O = P V.  Online softmax reaches this same result, so the oracle is the plain
 *     definition (no tiling, no running max).
 *
 * Readings where the pages are silent (each one also listed in the design notes):
 *   - softmax scale: a caller argument (the pages print the formula without one);
 *   - pool layout: key and value pools are separate, each [num_blocks][Hkv][block][D];
 *   - slot = physical_block * block_size + offset_in_block; a negative slot is skipped;
 *   - a query chunk of q_len rows over L keys sits at positions L-q_len .. L-1;
 *   - context length 0 gives a zero output.
 *
 * Precision: the pages fix bf16 storage (agentlenshq.com page, section "BF16"); they
 * fix no accumulation precision, so every sum here is in double, in index order, and
 * exp() is the C library's.  bf16 -> double is exact.
 *
 * Parity pins: every function here is checked by tests/test_oracle_*.py against
 * values fixed by the pages or by mathematics (block arithmetic, a hand-worked
 * block-table example, torch's scaled_dot_product_attention in float64, closed forms,
 * invariants); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Error codes returned by the oracle (0 = fine). */
#define PKO_OK 0
#define PKO_BAD_ARG 1
#define PKO_BAD_BLOCK 2 /* a block id outside [0, num_blocks) */
#define PKO_BAD_POSITION 3 /* a position beyond the block table or before 0 */

static double bf16_bits_to_double(uint16_t bits) {
  uint32_t word = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &word, sizeof f);
  return (double)f;
}

/* Number of 16-token (block_size) blocks a sequence of `tokens` tokens occupies:
 * blocks are added one at a time as tokens arrive ("vLLM", PagedAttention). */
int64_t pko_blocks_for_tokens(int64_t tokens, int32_t block_size) {
  if (tokens <= 0 || block_size <= 0) return 0;
  int64_t blocks = 0;
  int64_t capacity = 0;
  while (capacity < tokens) { /* add one block whenever the current ones are full */
    blocks += 1;
    capacity += block_size;
  }
  return blocks;
}

/* slot_mapping for the new tokens of every sequence ("Tiny-vLLM" Q&A: prepare_prefill /
 * prepare_decode).  Sequence s owns new tokens query_start_loc[s] .. query_start_loc[s+1]-1;
 * they are the last q_len of its context_lens[s] tokens.  Token at logical position p
 * lives in logical block p / block_size at offset p % block_size; the block table row
 * gives the physical block.  Bad entries produce slot -1 and an error code. */
int pko_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* context_lens, const int32_t* query_start_loc,
                     int32_t num_seqs, int32_t num_blocks, int32_t block_size,
                     int64_t* slot_mapping) {
  int err = PKO_OK;
  if (num_seqs < 0 || block_size <= 0) return PKO_BAD_ARG;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t first = query_start_loc[s];
    int32_t q_len = query_start_loc[s + 1] - first;
    for (int32_t i = 0; i < q_len; ++i) {
      int64_t pos = (int64_t)context_lens[s] - q_len + i;
      int64_t logical_block = pos / block_size;
      int64_t offset = pos % block_size;
      if (pos < 0 || logical_block >= max_blocks_per_seq) {
        slot_mapping[first + i] = -1;
        err = PKO_BAD_POSITION;
        continue;
      }
      int32_t phys = block_tables[(int64_t)s * max_blocks_per_seq + logical_block];
      if (phys < 0 || phys >= num_blocks) {
        slot_mapping[first + i] = -1;
        err = PKO_BAD_BLOCK;
        continue;
      }
      slot_mapping[first + i] = (int64_t)phys * block_size + offset;
    }
  }
  return err;
}

/* Element index of (physical block, kv head, offset in block, dim) in one pool. */
static int64_t pool_index(int64_t block, int32_t head, int64_t offset, int32_t dim,
                          int32_t num_kv_heads, int32_t block_size, int32_t head_dim) {
  return ((block * num_kv_heads + head) * block_size + offset) * head_dim + dim;
}

/* KV store ("reshape_and_cache"): write token t's key/value vectors (all heads) into the
 * slot slot_mapping[t]; negative slots are skipped.  A pure copy of the bf16 bits. */
int pko_reshape_and_cache(const uint16_t* key, const uint16_t* value,
                          const int64_t* slot_mapping, int32_t num_tokens,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, uint16_t* key_cache, uint16_t* value_cache) {
  int err = PKO_OK;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t block = slot / block_size;
    int64_t offset = slot % block_size;
    if (block >= num_blocks) {
      err = PKO_BAD_BLOCK;
      continue;
    }
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      for (int32_t d = 0; d < head_dim; ++d) {
        int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + d;
        int64_t dst = pool_index(block, h, offset, d, num_kv_heads, block_size, head_dim);
        key_cache[dst] = key[src];
        value_cache[dst] = value[src];
      }
    }
  }
  return err;
}

/* Block copy used by copy-on-write ("vLLM", PagedAttention: sequences that share a prompt
 * share its physical blocks and a block is copied only when one of them writes to it).
 * For each pair (src, dst) of block_mapping, every byte of block src (all kv heads, all
 * offsets, all dims) in both pools is copied to block dst, pairs in order. */
int pko_copy_blocks(uint16_t* key_cache, uint16_t* value_cache, int32_t num_blocks,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    const int64_t* block_mapping, int32_t num_pairs) {
  int err = PKO_OK;
  for (int32_t i = 0; i < num_pairs; ++i) {
    int64_t src = block_mapping[2 * i];
    int64_t dst = block_mapping[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      err = PKO_BAD_BLOCK;
      continue;
    }
    for (int32_t h = 0; h < num_kv_heads; ++h)
      for (int32_t off = 0; off < block_size; ++off)
        for (int32_t d = 0; d < head_dim; ++d) {
          int64_t from = pool_index(src, h, off, d, num_kv_heads, block_size, head_dim);
          int64_t to = pool_index(dst, h, off, d, num_kv_heads, block_size, head_dim);
          key_cache[to] = key_cache[from];
          value_cache[to] = value_cache[from];
        }
  }
  return err;
}

/* Gather the first `len` tokens of one sequence's kv head into contiguous double arrays
 * K[len][D], V[len][D] by walking its block table. */
static int gather_sequence(const uint16_t* key_cache, const uint16_t* value_cache,
                           int32_t num_blocks, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, const int32_t* table_row,
                           int32_t max_blocks_per_seq, int32_t len, int32_t kv_head,
                           double* K, double* V) {
  for (int32_t j = 0; j < len; ++j) {
    int32_t logical_block = j / block_size;
    int32_t offset = j % block_size;
    if (logical_block >= max_blocks_per_seq) return PKO_BAD_POSITION;
    int32_t phys = table_row[logical_block];
    if (phys < 0 || phys >= num_blocks) return PKO_BAD_BLOCK;
    for (int32_t d = 0; d < head_dim; ++d) {
      int64_t idx = pool_index(phys, kv_head, offset, d, num_kv_heads, block_size, head_dim);
      K[(int64_t)j * head_dim + d] = bf16_bits_to_double(key_cache[idx]);
      V[(int64_t)j * head_dim + d] = bf16_bits_to_double(value_cache[idx]);
    }
  }
  return PKO_OK;
}

/* Plain softmax attention of one query vector over keys 0..n_keys-1:
 * s_j = scale * sum_d q[d] K[j][d];  p_j = exp(s_j - max s) / sum_j exp(s_j - max s);
 * out[d] = sum_j p_j V[j][d].  n_keys == 0 gives zeros.  `scores` has room for n_keys. */
static void attend_one_query(const uint16_t* q_row, const double* K, const double* V,
                             int32_t n_keys, int32_t head_dim, double scale,
                             double* scores, double* out) {
  for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (n_keys <= 0) return;
  double m = -INFINITY;
  for (int32_t j = 0; j < n_keys; ++j) {
    double dot = 0.0;
    for (int32_t d = 0; d < head_dim; ++d)
      dot += bf16_bits_to_double(q_row[d]) * K[(int64_t)j * head_dim + d];
    scores[j] = scale * dot;
    if (scores[j] > m) m = scores[j];
  }
  double l = 0.0;
  for (int32_t j = 0; j < n_keys; ++j) {
    scores[j] = exp(scores[j] - m);
    l += scores[j];
  }
  for (int32_t j = 0; j < n_keys; ++j) {
    double p = scores[j] / l;
    for (int32_t d = 0; d < head_dim; ++d) out[d] += p * V[(int64_t)j * head_dim + d];
  }
}

/* Causal chunked attention over a paged prefix.  Sequence s has q_len =
 * query_start_loc[s+1] - query_start_loc[s] query rows that are the last q_len of its
 * context_lens[s] tokens; row i (position L - q_len + i) attends keys 0..L-q_len+i.
 * Query head h reads K/V head h / (num_q_heads / num_kv_heads).
 * q: bf16 [total_q][num_q_heads][head_dim];  out: double, same shape. */
int pko_prefill_chunk(double* out, const uint16_t* q, const int32_t* query_start_loc,
                      int32_t num_seqs, const uint16_t* key_cache,
                      const uint16_t* value_cache, int32_t num_blocks, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* context_lens,
                      int32_t num_q_heads, double scale) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return PKO_BAD_ARG;
  int32_t group = num_q_heads / num_kv_heads;
  int err = PKO_OK;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t first = query_start_loc[s];
    int32_t q_len = query_start_loc[s + 1] - first;
    int32_t L = context_lens[s];
    if (q_len <= 0) continue;
    if (L < q_len) {
      err = PKO_BAD_POSITION;
      continue;
    }
    size_t n = (size_t)(L > 0 ? L : 1) * head_dim;
    double* K = (double*)malloc(n * sizeof(double));
    double* V = (double*)malloc(n * sizeof(double));
    double* scores = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    if (!K || !V || !scores) {
      free(K); free(V); free(scores);
      return PKO_BAD_ARG;
    }
    for (int32_t g = 0; g < num_kv_heads; ++g) {
      int rc = gather_sequence(key_cache, value_cache, num_blocks, num_kv_heads, head_dim,
                               block_size, block_tables + (int64_t)s * max_blocks_per_seq,
                               max_blocks_per_seq, L, g, K, V);
      if (rc != PKO_OK) {
        err = rc;
        continue;
      }
      for (int32_t h = g * group; h < (g + 1) * group; ++h) {
        for (int32_t i = 0; i < q_len; ++i) {
          int64_t row = (int64_t)(first + i) * num_q_heads + h;
          int32_t visible = L - q_len + i + 1; /* keys 0 .. L-q_len+i */
          attend_one_query(q + row * head_dim, K, V, visible, head_dim, scale, scores,
                           out + row * head_dim);
        }
      }
    }
    free(K); free(V); free(scores);
  }
  return err;
}

/* Decode attention: one query (the newest token) per sequence over all context_lens[s]
 * cached tokens.  q: bf16 [num_seqs][num_q_heads][head_dim]; out: double, same shape. */
int pko_decode(double* out, const uint16_t* q, int32_t num_seqs, const uint16_t* key_cache,
               const uint16_t* value_cache, int32_t num_blocks, int32_t num_kv_heads,
               int32_t head_dim, int32_t block_size, const int32_t* block_tables,
               int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_q_heads,
               double scale) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return PKO_BAD_ARG;
  int32_t group = num_q_heads / num_kv_heads;
  int err = PKO_OK;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t L = context_lens[s];
    if (L < 0) {
      err = PKO_BAD_POSITION;
      continue;
    }
    size_t n = (size_t)(L > 0 ? L : 1) * head_dim;
    double* K = (double*)malloc(n * sizeof(double));
    double* V = (double*)malloc(n * sizeof(double));
    double* scores = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    if (!K || !V || !scores) {
      free(K); free(V); free(scores);
      return PKO_BAD_ARG;
    }
    for (int32_t g = 0; g < num_kv_heads; ++g) {
      int rc = gather_sequence(key_cache, value_cache, num_blocks, num_kv_heads, head_dim,
                               block_size, block_tables + (int64_t)s * max_blocks_per_seq,
                               max_blocks_per_seq, L, g, K, V);
      if (rc != PKO_OK) {
        err = rc;
        continue;
      }
      for (int32_t h = g * group; h < (g + 1) * group; ++h) {
        int64_t row = (int64_t)s * num_q_heads + h;
        attend_one_query(q + row * head_dim, K, V, L, head_dim, scale, scores,
                         out + row * head_dim);
      }
    }
    free(K); free(V); free(scores);
  }
  return err;
}
