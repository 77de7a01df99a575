// Host-side block manager: the "virtual memory" half of PagedAttention ("vLLM",
// blog.rlaisqls.com, section PagedAttention): a pool of fixed 16-token physical blocks, a
// per-sequence table from logical to physical blocks, blocks added one at a time as tokens
// arrive, blocks shared between sequences (beam search / parallel sampling) with reference
// counts, and copy-on-write when a sequence writes into a shared block.  Freed blocks return
// to the pool at once ("vLLM", section Continuous Batching: finished requests' slots are
// reclaimed immediately).
//
// Pure host code (no CUDA); the copies it decides are carried out by pa_copy_blocks.
#include <stdint.h>

#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

struct pa_block_manager {
  int32_t num_blocks;
  int32_t block_size;
  std::vector<int32_t> free_list;  // stack; the lowest ids are handed out first
  std::vector<int32_t> ref_count;
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t tokens = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;
};

namespace {

int64_t blocks_for(int64_t tokens, int32_t block_size) {
  return (tokens + block_size - 1) / block_size;
}

void release_block(pa_block_manager* bm, int32_t b) {
  if (--bm->ref_count[b] == 0) bm->free_list.push_back(b);
}

}  // namespace

extern "C" {

pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, pa_block_manager** out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return PA_ERR_INVALID_ARG;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->ref_count.assign(num_blocks, 0);
  bm->free_list.reserve(num_blocks);
  for (int32_t b = num_blocks - 1; b >= 0; --b) bm->free_list.push_back(b);
  *out = bm;
  return PA_OK;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int32_t pa_bm_num_free_blocks(const pa_block_manager* bm) {
  return bm ? static_cast<int32_t>(bm->free_list.size()) : -1;
}

int32_t pa_bm_ref_count(const pa_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref_count[block];
}

pa_status pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id) {
  if (!bm || seq_id < 0 || bm->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
  bm->seqs.emplace(seq_id, pa_block_manager::Seq());
  return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm || child < 0 || bm->seqs.count(child)) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq copy = it->second;  // shares every physical block
  for (int32_t b : copy.blocks) ++bm->ref_count[b];
  bm->seqs.emplace(child, std::move(copy));
  return PA_OK;
}

pa_status pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, int32_t num_tokens,
                              int64_t* cow_pairs, int32_t cow_capacity, int32_t* num_cow) {
  if (num_cow) *num_cow = 0;
  if (!bm || num_tokens < 0) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq& seq = it->second;
  if (num_tokens == 0) return PA_OK;
  const int64_t have = static_cast<int64_t>(seq.blocks.size());
  const int64_t need = blocks_for(seq.tokens + num_tokens, bm->block_size);
  // The new tokens land in the current last block when it is partly filled; if another
  // sequence shares that block it must be copied first.
  const bool writes_last = seq.tokens % bm->block_size != 0;
  const bool cow = writes_last && have > 0 && bm->ref_count[seq.blocks.back()] > 1;
  const int64_t fresh = (need - have) + (cow ? 1 : 0);
  if (fresh > static_cast<int64_t>(bm->free_list.size())) return PA_ERR_OUT_OF_BLOCKS;
  if (cow && (!cow_pairs || cow_capacity < 1)) return PA_ERR_INVALID_ARG;
  if (cow) {
    const int32_t shared = seq.blocks.back();
    const int32_t copy = bm->free_list.back();
    bm->free_list.pop_back();
    bm->ref_count[copy] = 1;
    --bm->ref_count[shared];  // still >= 1: the other sharers keep it
    seq.blocks.back() = copy;
    cow_pairs[0] = shared;
    cow_pairs[1] = copy;
    if (num_cow) *num_cow = 1;
  }
  for (int64_t i = have; i < need; ++i) {  // one block at a time, on demand
    const int32_t b = bm->free_list.back();
    bm->free_list.pop_back();
    bm->ref_count[b] = 1;
    seq.blocks.push_back(b);
  }
  seq.tokens += num_tokens;
  return PA_OK;
}

pa_status pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
  for (int32_t b : it->second.blocks) release_block(bm, b);
  bm->seqs.erase(it);
  return PA_OK;
}

int64_t pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : it->second.tokens;
}

int32_t pa_bm_block_table(const pa_block_manager* bm, int64_t seq_id, int32_t* out,
                          int32_t max_blocks) {
  if (!bm || (!out && max_blocks > 0)) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
  const auto& blocks = it->second.blocks;
  if (static_cast<int64_t>(blocks.size()) > max_blocks) return PA_ERR_INVALID_ARG;
  std::copy(blocks.begin(), blocks.end(), out);
  for (int32_t i = static_cast<int32_t>(blocks.size()); i < max_blocks; ++i) out[i] = -1;
  return static_cast<int32_t>(blocks.size());
}

}  // extern "C"
