// Causal chunked-prefill attention over a paged prefix, on tcgen05 tensor cores.
//
// What is computed ("vLLM", blog.rlaisqls.com, sections PagedAttention and Flash
// Attention; "tiny-vllm (1)", geonuchoi.com, sections 1 and 2): a sequence appends a chunk
// of q_len tokens to a context of L tokens (the chunk's own K/V already stored); chunk row
// i sits at position L - q_len + i and attends keys 0 .. L - q_len + i (causal mask) of
// its query head's K/V head (query head h reads K/V head h / 4), with an online softmax
// over key tiles so no score matrix reaches HBM.
//
// GB300 design.  QK^T and PV are dense contractions, so they run on the 5th-generation
// tensor cores with accumulators in tensor memory (TMEM):
//   * A work unit is one (32-token query tile, K/V head) of one sequence: 128 MMA rows =
//     32 tokens x 4 query heads sharing the K/V head (row = 4 * token + head), so each K/V
//     tile feeds four heads.
//   * Persistent grid, two CTAs per SM.  Every CTA first runs the same in-kernel plan: it
//     lists the (sequence, query tile) pairs, sorts them by their number of 64-key tiles,
//     heaviest first (a stable counting sort, identical in every CTA), and takes its share
//     of the units as a snake over that order, so the SMs end together.  (Batches beyond
//     the sort's size take the units in grid order instead.)  The CTA then serves its units
//     back to back: barrier phases, the K/V ring and the two S buffers carry over from one
//     unit to the next, the next unit's Q is loaded one unit ahead and written to TMEM
//     during the current unit's last tile, so its first scores are computed while the
//     current unit finishes.
//   * Warp 5 loads Q with one 3-D TMA box per unit (two Q buffers) and gathers every 64-key
//     K/V tile as four 16-row TMA boxes at the physical blocks named by the block table
//     (128-byte swizzle), into a 4-stage ring; the block table is read in prefetched
//     32-entry windows.
//   * Warp 4 (one thread) issues S = Q K^T (M128 N64 K64 into one of two fp32 S buffers,
//     so the next tile's scores are computed during this tile's softmax) and
//     [O | l] += P [V | 1] (M128 N80 K64, V read N-major): 16 extra columns of the B operand
//     come from a constant shared-memory atom of bf16 ones, one leading-byte offset from
//     each V slice, so the tensor core also accumulates the row sums l of exactly the bf16
//     P that weights V.  Both A operands come from TMEM: Q is copied there by the row warps
//     and P is written per tile over the first half of its own S buffer, so each MMA
//     streams only its K or V tile from shared memory.
//   * Warps 0-3 own one TMEM lane = one query row each: they read S, mask by absolute
//     position (diagonal tiles only), keep the running max in registers ([O | l] in TMEM is
//     rescaled only when the max grows by more than 2^8), write P as packed bf16 into TMEM,
//     and at the end of a unit divide O by l and store bf16 rows.
// TMEM per CTA (256 columns): S buffers 0..63 and 64..127 (P over 0..31 / 64..95), O
// 128..191, l 192..207, Q 224..255.
// Every mbarrier wait is bounded; on timeout the CTA records PA_DEVFLAG_TIMEOUT, drains
// its own copies and MMAs, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kGroup = 4;                         // query heads per K/V head
constexpr int kTokensPerTile = 32;
constexpr int kTileM = kTokensPerTile * kGroup;   // 128 MMA rows
constexpr int kTileN = 64;                        // keys per K/V tile
constexpr int kBlocksPerTile = kTileN / kBlockSize;
constexpr int kStages = 4;                        // K/V ring depth
constexpr int kQBytes = kTileM * kRowBytes;       // 16 KiB
constexpr int kKVBytes = kTileN * kRowBytes;      // 8 KiB per K (or V) tile
constexpr int kOnesBytes = 16 * kRowBytes;        // 16 key rows of bf16 1.0: the row-sum atom
constexpr int kMaxUnitsPerCta = 256;              // work units one CTA can hold in its list
constexpr int kSortThreads = 192;
constexpr int kMaxSortPairs = 2048;               // (sequence, query tile) pairs sorted in-kernel
constexpr int kSortBuckets = 64;
// Shared memory: Q x 2 | K ring | V ring | ones atom | barriers | misc | unit list.
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + 2 * kQBytes;
constexpr int kVOff = kKOff + kStages * kKVBytes;
constexpr int kOnesOff = kVOff + kStages * kKVBytes;
constexpr int kBarOff = kOnesOff + kOnesBytes;
constexpr int kNumBars = 2 + 2 + 2 * kStages + 2 + 2 + 1 + 1 + 1;  // 19
constexpr int kMiscOff = kBarOff + 24 * 8;
constexpr int kUnitOff = kMiscOff + 128;  // misc: TMEM address, abort flag, unit count, 24 ints of scratch
constexpr int kSmemBytes = kUnitOff + 2 * kMaxUnitsPerCta * 4;
static_assert(kNumBars <= 24, "barrier area");
static_assert(32 % kBlocksPerTile == 0, "block-table windows hold whole K/V tiles");
// The in-kernel sort uses the Q and K/V buffers as scratch before the pipeline starts.
constexpr int kSortScratchBytes = 4 * kMaxSortPairs * 4 + (1 + kSortThreads / 32) * kSortBuckets * 4;
static_assert(kSortScratchBytes <= kOnesOff, "sort scratch fits in the Q and K/V buffers");
// Two CTAs fit on one SM (2 x (kSmemBytes + 1 KiB reserved) <= 228 KiB, 2 x 256 TMEM
// columns = 512, <= 168 registers per thread), so one CTA's softmax overlaps the other's MMAs.
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kSCol = 0;     // two S buffers (fp32): columns 0..63 and 64..127; P (bf16
                                  // pairs) of a tile overwrites the first 32 of its S buffer
constexpr uint32_t kOCol = 128;   // O (fp32): columns 128..191, then 16 row-sum columns
constexpr uint32_t kLCol = kOCol + kHeadDim;  // row sum l (columns 192..207 hold 16 copies)
constexpr uint32_t kQCol = 224;   // Q (bf16 pairs): columns 224..255, the A operand of S = Q K^T
constexpr int kPVN = kHeadDim + 16;  // PV MMA width: 64 output dims + 16 ones columns
constexpr int kThreads = 192;
constexpr int kRowWarps = 4;  // barriers the row warps signal count one arrival per warp
constexpr float kRescaleThreshold = 8.0f;

struct PParams {
  __nv_bfloat16* out;
  const int32_t* query_start_loc;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t num_q_heads;
  float qk_scale;  // scale * log2(e)
  int32_t* status;
  int32_t num_query_tokens;
  int32_t num_seqs;
  int32_t q_tiles;  // query tiles of the longest chunk: ceil(max_query_len / 32)
  int32_t skip_single;  // 1: sequences with exactly one query row are served elsewhere
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* status) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  flag_error(status, PA_DEVFLAG_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// One work unit: query tile `tile` (32 tokens x 4 heads = 128 MMA rows) of sequence s against
// K/V head g, with everything the roles derive from it.
struct Unit {
  int s, g, tile;
  int q0, q_len, L;
  int tok0, ntok, keys, n_kv, blocks_needed;
};

// Whether sequence s has query rows to serve, and its rows / context.  Sequences with no rows
// are skipped silently; rows outside q / out or a context shorter than the chunk or longer
// than its block-table row are reported (when `report`) and skipped.
__device__ __forceinline__ bool sequence_ok(const PParams& p, int s, int* q0, int* q_len, int* L,
                                            bool report) {
  *q0 = p.query_start_loc[s];
  *q_len = p.query_start_loc[s + 1] - *q0;
  if (*q_len <= 0) return false;
  *L = p.context_lens[s];
  if (*q0 < 0 || *q0 + *q_len > p.num_query_tokens || *L < *q_len ||
      static_cast<int64_t>(*L) > static_cast<int64_t>(p.max_blocks_per_seq) * kBlockSize) {
    if (report) flag_error(p.status, PA_DEVFLAG_BAD_CONTEXT);
    return false;
  }
  return true;
}

__device__ __forceinline__ int tile_work(int L, int q_len, int tile) {
  const int ntok = min(kTokensPerTile, q_len - tile * kTokensPerTile);
  return (L - q_len + tile * kTokensPerTile + ntok + kTileN - 1) / kTileN;
}

__device__ __forceinline__ void fill_unit(Unit& u) {
  u.tok0 = u.tile * kTokensPerTile;
  u.ntok = min(kTokensPerTile, u.q_len - u.tok0);
  u.keys = u.L - u.q_len + u.tok0 + u.ntok;  // this tile needs keys 0 .. keys-1
  u.n_kv = (u.keys + kTileN - 1) / kTileN;
  u.blocks_needed = (u.keys + kBlockSize - 1) / kBlockSize;
}

// The CTA's sequence of work units.  Sorted mode: the units (every existing (sequence, query
// tile) pair x K/V head) were ordered heaviest first by the in-kernel plan, and this CTA's
// share (a snake over the order: round r takes position r*G + c, or r*G + G-1-c on odd
// rounds) sits in shared memory.  Otherwise (very large batches) units are taken in grid
// order, the query-tile index slowest and reversed, CTA c serving c, c + G, c + 2G, ...
struct Schedule {
  const int32_t* unit_s;   // shared memory (sorted mode)
  const int32_t* unit_tg;  // tile * 64 + g
  int n_units;             // sorted mode: this CTA's unit count; -1: grid order
};

__device__ __forceinline__ bool next_unit(const PParams& p, const Schedule& sc, int& k, Unit& u) {
  if (sc.n_units >= 0) {
    if (k >= sc.n_units) return false;
    u.s = sc.unit_s[k];
    const int tg = sc.unit_tg[k];
    u.tile = tg >> 6;
    u.g = tg & 63;
    ++k;
    sequence_ok(p, u.s, &u.q0, &u.q_len, &u.L, false);
    fill_unit(u);
    return true;
  }
  const int64_t per_tile = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads;
  const int64_t total = per_tile * p.q_tiles;
  for (;;) {
    const int64_t x = blockIdx.x + static_cast<int64_t>(k) * gridDim.x;
    if (x >= total) return false;
    ++k;
    const int64_t rem = x % per_tile;
    u.tile = p.q_tiles - 1 - static_cast<int>(x / per_tile);
    u.g = static_cast<int>(rem / p.num_seqs);
    u.s = static_cast<int>(rem % p.num_seqs);
    if (!sequence_ok(p, u.s, &u.q0, &u.q_len, &u.L, u.tile == 0 && u.g == 0)) continue;
    if (u.tile * kTokensPerTile >= u.q_len || (p.skip_single && u.q_len == 1)) continue;
    fill_unit(u);
    return true;
  }
}

// Exclusive block-wide prefix sum over kSortThreads values; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += x;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kSortThreads / 32; ++w) {
    const int x = scratch[w];
    if (w < warp) before += x;
    all += x;
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

// In-kernel plan, run by every CTA on the same inputs (so every CTA derives the same order):
// list the (sequence, query tile) pairs, sort them by their number of 64-key tiles, heaviest
// first (a stable counting sort on 64 buckets: ranks within a bucket come from warp matches
// in pair order, 192 pairs per round), and take this CTA's units.  Returns the unit count, or
// -1 when the batch has more pairs than the sort handles (grid order then).
__device__ int plan_units(const PParams& p, uint8_t* scratch, int* red, int32_t* unit_s,
                          int32_t* unit_tg) {
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int kWarpsP = kSortThreads / 32;
  int* pair_s = reinterpret_cast<int*>(scratch);  // [kMaxSortPairs]
  int* pair_t = pair_s + kMaxSortPairs;
  int* pair_w = pair_t + kMaxSortPairs;
  int* sorted = pair_w + kMaxSortPairs;
  int* base = sorted + kMaxSortPairs;              // [kSortBuckets] next position per bucket
  int* wcnt = base + kSortBuckets;                 // [kWarpsP][kSortBuckets] per-round counts
  // 1. enumerate the pairs, 192 sequences at a time
  int n = 0;
  for (int s0 = 0; s0 < p.num_seqs; s0 += kSortThreads) {
    const int s = s0 + tid;
    int q0 = 0, q_len = 0, L = 0, tiles = 0;
    if (s < p.num_seqs && sequence_ok(p, s, &q0, &q_len, &L, blockIdx.x == 0) &&
        !(p.skip_single && q_len == 1))
      tiles = (q_len + kTokensPerTile - 1) / kTokensPerTile;
    int total;
    const int excl = block_exclusive_scan(tiles, red, &total);
    if (n + total <= kMaxSortPairs) {
      for (int t = 0; t < tiles; ++t) {
        pair_s[n + excl + t] = s;
        pair_t[n + excl + t] = t;
        pair_w[n + excl + t] = tile_work(L, q_len, t);
      }
    }
    n += total;
  }
  const int units = n * p.num_kv_heads;
  const int G = gridDim.x;
  if (n > kMaxSortPairs || (units + G - 1) / G > kMaxUnitsPerCta) return -1;
  for (int i = tid; i < kSortBuckets * (kWarpsP + 1); i += kSortThreads) base[i] = 0;  // + wcnt
  __syncthreads();  // the pairs written above are read by other threads below
  // 2. largest work, then bucket = work scaled to 0..63 (heavier = higher)
  int wmax = 0;
  for (int i = tid; i < n; i += kSortThreads) wmax = max(wmax, pair_w[i]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, d));
  if (lane == 0) red[8 + warp] = wmax;
  __syncthreads();
  wmax = 0;
  for (int w = 0; w < kWarpsP; ++w) wmax = max(wmax, red[8 + w]);
  auto bucket = [&](int i) {
    const int b = static_cast<int>((static_cast<int64_t>(pair_w[i]) * kSortBuckets) / (wmax + 1));
    return min(max(b, 0), kSortBuckets - 1);
  };
  for (int i = tid; i < n; i += kSortThreads) atomicAdd(&base[bucket(i)], 1);
  __syncthreads();
  // 3. bucket starts, heaviest bucket first (one warp, two buckets per lane)
  if (warp == 0) {
    const int hi = base[kSortBuckets - 1 - 2 * lane], lo = base[kSortBuckets - 2 - 2 * lane];
    int incl = hi + lo;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += x;
    }
    const int start = incl - hi - lo;
    base[kSortBuckets - 1 - 2 * lane] = start;
    base[kSortBuckets - 2 - 2 * lane] = start + hi;
  }
  __syncthreads();
  // 4. stable placement, pair i = round * 192 + tid: its rank in its bucket counts the pairs of
  // earlier rounds (base), of earlier warps in this round (wcnt) and of lower lanes (match)
  for (int r0 = 0; r0 < n; r0 += kSortThreads) {
    const int i = r0 + tid;
    const int b = i < n ? bucket(i) : kSortBuckets;  // kSortBuckets: no pair
    const unsigned same = __match_any_sync(0xffffffffu, b);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (b < kSortBuckets && rank == 0) wcnt[warp * kSortBuckets + b] = __popc(same);
    __syncthreads();
    if (b < kSortBuckets) {
      int before = base[b] + rank;
      for (int w = 0; w < warp; ++w) before += wcnt[w * kSortBuckets + b];
      sorted[before] = i;
    }
    __syncthreads();
    if (tid < kSortBuckets) {
      int add = 0;
      for (int w = 0; w < kWarpsP; ++w) {
        add += wcnt[w * kSortBuckets + tid];
        wcnt[w * kSortBuckets + tid] = 0;
      }
      base[tid] += add;
    }
    __syncthreads();
  }
  // 5. this CTA's units: a snake over the sorted order, K/V head fastest
  const int c = blockIdx.x;
  const int rounds = (units + G - 1) / G;
  int mine = 0;
  for (int r = 0; r < rounds; ++r) {
    const int pos = r * G + ((r & 1) ? G - 1 - c : c);
    if (pos < units) ++mine;
  }
  for (int k = tid; k < mine; k += kSortThreads) {
    const int pos = k * G + ((k & 1) ? G - 1 - c : c);
    const int pr = sorted[pos / p.num_kv_heads];
    unit_s[k] = pair_s[pr];
    unit_tg[k] = pair_t[pr] * 64 + pos % p.num_kv_heads;
  }
  return mine;
}

// Persistent causal chunk attention: each CTA serves its work units one after the other,
// with the barrier phases, the K/V ring and the two S buffers carried across units (tile
// counter jt counts every 64-key tile this CTA has processed).
__global__ void __launch_bounds__(kThreads, 2)
paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const PParams p) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // A decode launch that follows with programmatic dependent launch may start its
  // prologue as this grid's CTAs leave the SMs (it waits for this grid before touching what
  // this grid writes).  When this grid itself was launched that way (the unified varlen
  // launch, behind the decode of the same batch, whose outputs and inputs it does not
  // touch), it waits for that grid only at its end, so that its completion still implies
  // the previous grid's.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  extern __shared__ __align__(1024) uint8_t smem[];  // 128-byte swizzle atoms need 1 KiB
  if ((smem_addr(smem) & 1023u) != 0) {  // never issue swizzled copies to a misaligned tile
    if (tid == 0) flag_error(p.status, PA_DEVFLAG_LAYOUT);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }
  uint8_t* sq = smem + kQOff;  // two Q buffers
  uint8_t* sk = smem + kKOff;
  uint8_t* sv = smem + kVOff;
  uint8_t* sones = smem + kOnesOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars;         // [2] Q tile landed in buffer b
  uint64_t* q_empty = bars + 2;    // [2] Q buffer b copied into tensor memory
  uint64_t* kv_full = bars + 4;    // [kStages]
  // pv_done[st]: the P V of the tile held in stage st has completed.  One commit serves
  // two readers: the producer (the stage may be refilled) and the row warps (O and its row
  // sum are up to date).  Tile jt is phase jt / kStages of pv_done[jt % kStages].
  uint64_t* pv_done = kv_full + kStages;
  uint64_t* s_ready = pv_done + kStages;  // [2]
  // p_ready[b]: P of the tile in S buffer b is in tensor memory (phase jt / 2 for tile jt).
  // Per buffer, so the issuing thread can never fall two phases behind: P(jt+2) needs
  // S(jt+2), which is issued only after the wait for P(jt).
  uint64_t* p_ready = s_ready + 2;
  uint64_t* o_free = p_ready + 2;  // the epilogue has read O out of tensor memory
  uint64_t* q_tmem = o_free + 1;   // this unit's Q is in tensor memory
  uint64_t* drain = q_tmem + 1;
  int* misc = reinterpret_cast<int*>(smem + kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int& abort_flag = *reinterpret_cast<volatile int*>(misc + 1);
  int* n_units_s = misc + 2;
  int* red = misc + 4;  // 24 ints of scan / reduction scratch (red[0..5], red[8..13] used)
  int32_t* unit_s = reinterpret_cast<int32_t*>(smem + kUnitOff);
  int32_t* unit_tg = unit_s + kMaxUnitsPerCta;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], kRowWarps);
      mbar_init(&s_ready[b], 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&p_ready[0], kRowWarps);
    mbar_init(&p_ready[1], kRowWarps);
    mbar_init(o_free, kRowWarps);
    mbar_init(q_tmem, kRowWarps);
    mbar_init(drain, 1);
    fence_barrier_init();
    abort_flag = 0;
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 5 && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  // The plan (in the Q and K/V buffers, before any copy lands there).
  const int n_units = plan_units(p, smem, red, unit_s, unit_tg);
  if (tid == 0) *n_units_s = n_units;
  // The ones atom: every bf16 of it is 1.0, so the 16 extra columns of O += P [V | 1] each
  // accumulate the row sum of P, exactly the bf16 values that weight V.
  for (int i = tid; i < kOnesBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(sones)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async_smem();  // generic writes (plan scratch, ones) before async-proxy access
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  Schedule sc;
  sc.unit_s = unit_s;
  sc.unit_tg = unit_tg;
  sc.n_units = *n_units_s;

  if (warp == 5) {
    // ================================ TMA producer ================================
    int k = 0;
    Unit cur, nxt;
    bool have = next_unit(p, sc, k, cur);
    bool have_next = have && next_unit(p, sc, k, nxt);
    int nq = 0;  // Q tiles issued
    auto load_q = [&](const Unit& u) {
      const int b = nq & 1;
      bool ok = true;
      if (lane == 0) {
        if (nq >= 2)  // buffer b held the Q of unit nq-2: wait until it is in tensor memory
          ok = wait_or_abort(&q_empty[b], static_cast<uint32_t>(((nq - 2) >> 1) & 1), &abort_flag,
                             p.status);
        if (ok) {
          mbar_arrive_expect_tx(&q_full[b], kQBytes);
          tma_load_3d(sq + b * kQBytes, &tmap_q, 0, u.g * kGroup, u.q0 + u.tok0, &q_full[b]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok) ++nq;
      return ok;
    };
    bool ok = !have || load_q(cur);
    int jt = 0;  // K/V tiles issued
    while (ok && have) {
      if (have_next && !(ok = load_q(nxt))) break;  // the next unit's Q, one unit ahead
      const int32_t* row = p.block_tables + static_cast<int64_t>(cur.s) * p.max_blocks_per_seq;
      // The block table is read 32 entries (eight K/V tiles) at a time, one entry per lane,
      // with the next window already in flight, so no tile waits on a block-table load.
      auto fetch = [&](int base) -> int32_t {
        return base + lane < cur.blocks_needed ? __ldg(row + base + lane) : 0;
      };
      int win_base = 0;
      int32_t win = fetch(0);
      int32_t win_next = fetch(32);
      for (int j = 0; j < cur.n_kv; ++j, ++jt) {
        const int st = jt % kStages;
        const int lb0 = j * kBlocksPerTile;
        if (lb0 >= win_base + 32) {
          win_base += 32;
          win = win_next;
          win_next = fetch(win_base + 32);
        }
        const int lb = lb0 + lane;
        const bool need = lane < kBlocksPerTile && lb < cur.blocks_needed;
        const int32_t entry =
            __shfl_sync(0xffffffffu, win, (lb0 - win_base) + (lane & (kBlocksPerTile - 1)));
        const int32_t phys = need ? entry : 0;
        const bool bad = need && (phys < 0 || phys >= p.num_blocks);
        const bool load = need && !bad;
        const unsigned mask = __ballot_sync(0xffffffffu, load);
        const unsigned bad_mask = __ballot_sync(0xffffffffu, bad);
        if (lane == 0 && bad_mask != 0) flag_error(p.status, PA_DEVFLAG_BAD_BLOCK);
        int go = 1;
        if (lane == 0) {
          go = wait_or_abort(&pv_done[st], static_cast<uint32_t>((jt / kStages) & 1) ^ 1u,
                             &abort_flag, p.status);
          if (go) mbar_arrive_expect_tx(&kv_full[st], __popc(mask) * 2u * kTileBytes);
        }
        go = __shfl_sync(0xffffffffu, go, 0);
        if (!go) {
          ok = false;
          break;
        }
        if (load) {
          const int y = (phys * p.num_kv_heads + cur.g) * kBlockSize;
          tma_load_2d(sk + st * kKVBytes + lane * kTileBytes, &tmap_k, 0, y, &kv_full[st]);
          tma_load_2d(sv + st * kKVBytes + lane * kTileBytes, &tmap_v, 0, y, &kv_full[st]);
        }
      }
      cur = nxt;
      have = have_next;
      if (have) have_next = next_unit(p, sc, k, nxt);
    }
    // leave no copy in flight: wait (bounded) for the last Q of each buffer and the last
    // fill of each stage
    if (lane == 0) {
      for (int b = 0; b < 2 && b < nq; ++b) {
        const int last = b + ((nq - 1 - b) / 2) * 2;
        if (!mbar_wait(&q_full[b], static_cast<uint32_t>((last >> 1) & 1)))
          flag_error(p.status, PA_DEVFLAG_TIMEOUT);
      }
      for (int st = 0; st < kStages && st < jt; ++st) {
        const int last = st + ((jt - 1 - st) / kStages) * kStages;
        if (!mbar_wait(&kv_full[st], static_cast<uint32_t>((last / kStages) & 1)))
          flag_error(p.status, PA_DEVFLAG_TIMEOUT);
      }
    }
  } else if (warp == 4) {
    // ================================ MMA issuer ==================================
    // Both A operands live in tensor memory (Q copied there once per unit, P written there by
    // the row warps over its tile's scores), so each MMA streams only its B tile (K or V,
    // 2 KiB per K16 step) from shared memory.  Order: S(0), S(1), PV(0), S(2), PV(1), ...
    // over the CTA's tiles of all its units: the scores of the next tile (of this unit or
    // the next) are on the tensor core while the row warps run the softmax of the current
    // one; S(j+2) reuses the buffer of P(j) only after PV(j) (one thread's MMAs complete in
    // order).
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTileM, kTileN, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kTileM, kPVN, true);
      const uint32_t ones_addr = smem_addr(sones);
      auto issue_s = [&](int jt) -> bool {
        const int st = jt % kStages;
        if (!wait_or_abort(&kv_full[st], static_cast<uint32_t>((jt / kStages) & 1), &abort_flag,
                           p.status))
          return false;
        tc_fence_after_sync();
        // K16 step kk starts 32 bytes further into each 128-byte swizzled row: +2 in the
        // descriptor's start-address field (16-byte units; no carry for shared addresses)
        const uint64_t k_desc = sw128_desc(smem_addr(sk + st * kKVBytes), 16, 1024);
        const uint32_t s_tmem = tmem + kSCol + (jt & 1) * kTileN;
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          umma_bf16_ts(s_tmem, tmem + kQCol + kk * 8, k_desc + 2 * kk, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_ready[jt & 1]);
        return true;
      };
      auto issue_pv = [&](int jt, bool first) {
        const uint32_t v_base = smem_addr(sv + (jt % kStages) * kKVBytes);
        const uint32_t p_tmem = tmem + kSCol + (jt & 1) * kTileN;
        // B = [V rows kk*16 .. +15 | ones]: output dims 0..63 from the V tile (N-major,
        // 128-byte swizzle), columns 64..79 from the ones atom, one leading-byte offset away.
        // Step kk starts 2 KiB further (+128 in the start-address field) and its leading-byte
        // offset to the ones atom is 2 KiB shorter (-128 in that field, bits 16..29).
        const uint64_t v_desc = sw128_desc(v_base, ones_addr - v_base, 1024);
        constexpr uint64_t kStep = (uint64_t{1} << 7) - (uint64_t{1} << 23);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          umma_bf16_ts(tmem + kOCol, p_tmem + kk * 8, v_desc + kk * kStep, kIdescO,
                       (!first || kk > 0) ? 1u : 0u);
        }
        umma_commit(&pv_done[jt % kStages]);
      };
      int k = 0;
      Unit cur, nxt;
      bool have = next_unit(p, sc, k, cur);
      bool have_next = have && next_unit(p, sc, k, nxt);
      bool ok = have && wait_or_abort(q_tmem, 0, &abort_flag, p.status);
      if (ok) {
        tc_fence_after_sync();
        ok = issue_s(0);
      }
      int jt = 0, kq = 0;
      while (ok && have) {
        for (int j = 0; ok && j < cur.n_kv; ++j, ++jt) {
          if (j + 1 < cur.n_kv) {
            ok = issue_s(jt + 1);
          } else if (have_next) {  // the next unit's first scores: its Q must be in TMEM
            ok = wait_or_abort(q_tmem, static_cast<uint32_t>((kq + 1) & 1), &abort_flag, p.status);
            if (ok) {
              tc_fence_after_sync();
              ok = issue_s(jt + 1);
            }
          }
          if (!ok) break;
          if (!(ok = wait_or_abort(&p_ready[jt & 1], static_cast<uint32_t>((jt >> 1) & 1),
                                   &abort_flag, p.status)))
            break;
          if (j == 0 && kq > 0) {  // O is overwritten: the last unit's epilogue has read it
            if (!(ok = wait_or_abort(o_free, static_cast<uint32_t>((kq - 1) & 1), &abort_flag,
                                     p.status)))
              break;
          }
          tc_fence_after_sync();
          issue_pv(jt, j == 0);
        }
        cur = nxt;
        have = have_next;
        if (have) have_next = next_unit(p, sc, k, nxt);
        ++kq;
      }
      // wait (bounded) until every MMA issued above has completed
      umma_commit(drain);
      if (!mbar_wait(drain, 0)) flag_error(p.status, PA_DEVFLAG_TIMEOUT);
    }
  } else {
    // ============================ softmax / epilogue (warps 0-3) ============================
    const int r = tid;  // MMA row == TMEM lane
    const int tt = r >> 2;
    const int hh = r & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int k = 0;
    Unit cur, nxt;
    bool have = next_unit(p, sc, k, cur);
    bool have_next = have && next_unit(p, sc, k, nxt);
    int kq = 0;  // units started
    // copy this row of Q (unit kq, buffer kq & 1, 128-byte swizzled) into tensor memory
    auto copy_q = [&](int kq_) -> bool {
      const int b = kq_ & 1;
      bool ok = wait_or_abort(&q_full[b], static_cast<uint32_t>((kq_ >> 1) & 1), &abort_flag,
                              p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return false;
      uint32_t qv[32];
      const uint8_t* qrow = sq + b * kQBytes + r * kRowBytes;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 x = lds128(qrow + ((c ^ (r & 7)) * 16));
        qv[4 * c] = x.x;
        qv[4 * c + 1] = x.y;
        qv[4 * c + 2] = x.z;
        qv[4 * c + 3] = x.w;
      }
      tmem_st32(lane_addr + kQCol, qv);
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();  // every lane's tensor-memory store and fence precede the warp's arrival
      if (lane == 0) {
        mbar_arrive(&q_empty[b]);
        mbar_arrive(q_tmem);
      }
      return true;
    };
    bool ok = !have || copy_q(0);
    int jt = 0;
    while (ok && have) {
      const int token = cur.tok0 + tt;
      const bool row_ok = token < cur.q_len;
      const int pos = cur.L - cur.q_len + min(token, cur.q_len - 1);
      const int pos_lo = cur.L - cur.q_len + cur.tok0;  // smallest position among the rows
      float m = -INFINITY;
      for (int j = 0; j < cur.n_kv; ++j, ++jt) {
        ok = wait_or_abort(&s_ready[jt & 1], static_cast<uint32_t>((jt >> 1) & 1), &abort_flag,
                           p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();
        const int kb = j * kTileN;
        const uint32_t s_addr = lane_addr + kSCol + (jt & 1) * kTileN;
        uint32_t v[2][32];  // raw scores; then, in place in v[0], packed bf16 probabilities
        tmem_ld32(s_addr, v[0]);
        tmem_ld32(s_addr + 32, v[1]);
        tmem_wait_ld();
        if (j == cur.n_kv - 1 && have_next) {
          // every score MMA of this unit has completed: the next unit's Q may replace it
          if (!(ok = copy_q(kq + 1))) break;
        }
        if (kb + kTileN - 1 > pos_lo) {
          // a tile on the causal diagonal (uniform over the CTA): hide keys past each row's
          // position before the maximum; exp2(-inf) = 0 then drops them from P and the sum
#pragma unroll
          for (int i = 0; i < kTileN; ++i)
            if (kb + i > pos) v[i >> 5][i & 31] = __float_as_uint(-INFINITY);
        }
        // tile maximum of the raw scores (the scale is positive, so it commutes with max)
        float mx[4];
#pragma unroll
        for (int a4 = 0; a4 < 4; ++a4) {
          mx[a4] = __uint_as_float(v[a4 >> 1][16 * (a4 & 1)]);
#pragma unroll
          for (int i = 1; i < 16; i += 2)
            mx[a4] = max3f(mx[a4], __uint_as_float(v[a4 >> 1][16 * (a4 & 1) + i]),
                           __uint_as_float(v[a4 >> 1][16 * (a4 & 1) + i + 1]));
        }
        const float mt = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * p.qk_scale;
        const float m_new = fmaxf(m, mt);
        const bool grow = m_new - m > kRescaleThreshold;  // true on the first tile (m = -inf)
        float alpha = 1.f;
        if (grow) {
          alpha = fast_exp2(m - m_new);
          m = m_new;
        }
        // p = 2^(s * scale - m) two at a time, packed to bf16 into v[0] (the row sum comes
        // from the tensor core's ones columns)
        const float2 qs2 = make_float2(p.qk_scale, p.qk_scale);
        const float2 nm2 = make_float2(-m, -m);
#pragma unroll
        for (int i = 0; i < kTileN / 2; ++i) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(v[i >> 4][(2 * i) & 31]),
                                                  __uint_as_float(v[i >> 4][(2 * i + 1) & 31])),
                                      qs2, nm2);
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(fast_exp2(x.x), fast_exp2(x.y));
          v[0][i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        if (j == cur.n_kv - 1 && kb + kTileN > cur.keys) {
          // V rows past the last needed key are never weighted, but may hold NaN (unused
          // slots) or stale data: zero them so 0 * V stays 0 in the tensor core.
          if (r < kTileN && kb + r >= cur.keys) {
            uint4* vrow = reinterpret_cast<uint4*>(sv + (jt % kStages) * kKVBytes + r * kRowBytes);
#pragma unroll
            for (int i = 0; i < kRowBytes / 16; ++i) vrow[i] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // O and its row sum are rescaled once PV(jt-1) is done with them.  Only a rescale
          // waits for it: P(jt) itself overwrites its own S buffer, whose last reader PV(jt-2)
          // completed before S(jt) did.  Skipping the wait on other tiles is safe because
          // the barrier is per stage: its previous phase (PV(jt-5)) was observed by the
          // producer before tile jt-1 was loaded, and its next one needs P(jt+3), so the
          // parity wait below cannot alias a phase two away.
          ok = wait_or_abort(&pv_done[(jt - 1) % kStages],
                             static_cast<uint32_t>(((jt - 1) / kStages) & 1), &abort_flag, p.status);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after_sync();
          uint32_t(&o)[32] = v[1];  // the raw scores there are spent
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            tmem_ld32(lane_addr + kOCol + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = __fmul2_rn(
                  make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), a2);
              o[2 * i] = __float_as_uint(x.x);
              o[2 * i + 1] = __float_as_uint(x.y);
            }
            tmem_st32(lane_addr + kOCol + 32 * c, o);
          }
          const uint32_t lsum = tmem_ld1(lane_addr + kLCol);
          tmem_wait_ld();
          tmem_st1(lane_addr + kLCol, __float_as_uint(__uint_as_float(lsum) * alpha));
        }
        tmem_st32(lane_addr + kSCol + (jt & 1) * kTileN, v[0]);  // P(jt) over S(jt)
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[jt & 1]);
      }
      if (!ok) break;
      // ---- epilogue: O / l of this unit, then release O to the next unit's first PV ----
      ok = wait_or_abort(&pv_done[(jt - 1) % kStages],
                         static_cast<uint32_t>(((jt - 1) / kStages) & 1), &abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t o[2][32];
      tmem_ld32(lane_addr + kOCol, o[0]);
      tmem_ld32(lane_addr + kOCol + 32, o[1]);
      const uint32_t lsum = tmem_ld1(lane_addr + kLCol);
      tmem_wait_ld();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      const float inv = 1.f / __uint_as_float(lsum);  // l >= 1: the max key weighs >= 1
      if (row_ok) {
        __nv_bfloat16* dst = p.out + (static_cast<int64_t>(cur.q0 + token) * p.num_q_heads +
                                      cur.g * kGroup + hh) * kHeadDim;
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = q8 * 8 + 2 * e;
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                __uint_as_float(o[i >> 5][i & 31]) * inv, __uint_as_float(o[i >> 5][(i + 1) & 31]) * inv);
            w[e] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(dst + 8 * q8) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      cur = nxt;
      have = have_next;
      if (have) have_next = next_unit(p, sc, k, nxt);
      ++kq;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

// [rows][64] bf16 tensor read in boxes of `box_rows` rows (128-byte swizzle); also the
// decode kernel's view of the pools.
bool encode_pool_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// q as [tokens][heads][64]; one box = 32 tokens x 4 heads (the 128 MMA rows of a tile).
bool encode_q(CUtensorMap* map, const void* base, uint64_t tokens, uint64_t heads) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), heads, tokens};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes), heads * kRowBytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), kGroup, kTokensPerTile};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

// Shared set-up of both launch forms: kernel attributes, tensor maps, parameters.
cudaError_t prepare(const PrefillArgs& a, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv,
                    PParams* p) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const uint64_t pool_rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  if (pool_rows >= (1ull << 31)) return cudaErrorInvalidValue;
  if (!encode_q(tq, a.q, static_cast<uint64_t>(a.num_query_tokens), a.num_q_heads) ||
      !encode_pool_rows(tk, a.key_cache, pool_rows, kBlockSize) ||
      !encode_pool_rows(tv, a.value_cache, pool_rows, kBlockSize))
    return cudaErrorInvalidValue;
  p->out = static_cast<__nv_bfloat16*>(a.out);
  p->query_start_loc = a.query_start_loc;
  p->block_tables = a.block_tables;
  p->max_blocks_per_seq = a.max_blocks_per_seq;
  p->context_lens = a.context_lens;
  p->num_blocks = a.num_blocks;
  p->num_kv_heads = a.num_kv_heads;
  p->num_q_heads = a.num_q_heads;
  p->qk_scale = a.scale * 1.4426950408889634f;
  p->status = a.status;
  p->num_query_tokens = a.num_query_tokens;
  p->num_seqs = a.num_seqs;
  p->q_tiles = (a.max_query_len + kTokensPerTile - 1) / kTokensPerTile;
  p->skip_single = 0;
  return cudaSuccess;
}

}  // namespace

namespace {

cudaError_t launch_prefill_kernel(const PrefillArgs& a, bool skip_single, cudaStream_t stream,
                                  bool overlap_previous = false, int32_t max_sms = 0) {
  CUtensorMap tq, tk, tv;
  PParams p;
  cudaError_t e = prepare(a, &tq, &tk, &tv, &p);
  if (e != cudaSuccess) return e;
  p.skip_single = skip_single ? 1 : 0;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if (max_sms > 0 && max_sms < sms) sms = max_sms;
  // persistent: two CTAs per SM, never more CTAs than work units can exist
  const int64_t units_upper = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads * p.q_tiles;
  const int64_t grid = units_upper < 2LL * sms ? units_upper : 2LL * sms;
  if (grid < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap_previous ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, paged_prefill_kernel, tq, tk, tv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Decode plan of a mixed batch's one-row sequences: a balanced split over the device, every
// context bounded by its block-table row.
cudaError_t varlen_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                               int32_t max_blocks_per_seq, DecodePlan* plan,
                               int32_t max_sms = 0) {
  const int64_t max_ctx = static_cast<int64_t>(max_blocks_per_seq) * kBlockSize;
  return plan_decode(num_seqs, num_kv_heads, num_q_heads,
                     static_cast<int32_t>(max_ctx < 0x7fffffff ? max_ctx : 0x7fffffff), 0, plan,
                     max_sms);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream, bool overlap_previous,
                           int32_t max_sms) {
  return launch_prefill_kernel(a, false, stream, overlap_previous, max_sms);
}

bool varlen_routes_decode_rows(int32_t num_seqs) { return num_seqs <= decode_max_seqs(); }

size_t varlen_workspace_need(const PrefillArgs& a) {
  if (!varlen_routes_decode_rows(a.num_seqs)) return 16;
  DecodePlan plan;
  if (varlen_decode_plan(a.num_seqs, a.num_kv_heads, a.num_q_heads, a.max_blocks_per_seq,
                         &plan) != cudaSuccess)
    return 0;
  return plan.workspace_bytes;
}

size_t varlen_workspace_size(int32_t num_seqs, int32_t num_query_tokens) {
  (void)num_query_tokens;
  if (!varlen_routes_decode_rows(num_seqs)) return 16;
  // an upper bound for any head count (64 K/V heads) and context length
  DecodePlan plan;
  if (plan_decode(num_seqs, 64, 256, 0x7fffffff, 0, &plan) != cudaSuccess) return 0;
  return plan.workspace_bytes;
}

cudaError_t launch_varlen(const PrefillArgs& a, void* workspace, cudaStream_t stream,
                          int32_t decode_sms) {
  if (!varlen_routes_decode_rows(a.num_seqs))  // every row on the tensor-core kernel
    return launch_prefill_kernel(a, false, stream);
  // decode_sms in 1 .. SMs-1: the decode rows on that many SMs, the chunks beside them on
  // the others at the same time
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool split = decode_sms > 0 && decode_sms < sms;
  // Decode rows (q_len 1) on the CUDA-core decode kernel, reading and writing their rows in
  // place; its workspace counters start at zero (cleared on the stream, nothing allocated).
  DecodePlan plan;
  e = varlen_decode_plan(a.num_seqs, a.num_kv_heads, a.num_q_heads, a.max_blocks_per_seq, &plan,
                         split ? decode_sms : 0);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(static_cast<uint8_t*>(workspace) + plan.ws_count_offset, 0,
                      plan.ws_meta_bytes - plan.ws_count_offset, stream);
  if (e != cudaSuccess) return e;
  DecodeArgs d;
  d.out = a.out;
  d.q = a.q;
  d.key_cache = a.key_cache;
  d.value_cache = a.value_cache;
  d.block_tables = a.block_tables;
  d.max_blocks_per_seq = a.max_blocks_per_seq;
  d.context_lens = a.context_lens;
  d.num_seqs = a.num_seqs;
  d.num_q_heads = a.num_q_heads;
  d.num_kv_heads = a.num_kv_heads;
  d.num_blocks = a.num_blocks;
  d.scale = a.scale;
  d.workspace = workspace;
  d.status = a.status;
  d.q_rows = a.query_start_loc;
  d.num_query_tokens = a.num_query_tokens;
  e = launch_decode(d, plan, stream);
  if (e != cudaSuccess) return e;
  // Chunks (q_len > 1) on the tensor-core kernel; none can exist when the host bound of
  // q_len is 1 (a decode-only batch), and then nothing more is launched.
  if (a.max_query_len <= 1) return cudaSuccess;
  // The chunk launch reads nothing the decode launch writes and writes other rows, so it
  // may start as the decode's CTAs leave, or at once on the SMs the decode leaves free (it
  // waits for the decode grid before it ends).
  return launch_prefill_kernel(a, true, stream, /*overlap_previous=*/true,
                               split ? sms - decode_sms : 0);
}

}  // namespace pkv
