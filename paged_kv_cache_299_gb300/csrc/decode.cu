// Paged decode attention with online softmax and a balanced split-KV merge.
//
// What is computed ("vLLM", blog.rlaisqls.com, sections PagedAttention and Flash
// Attention; "tiny-vllm (1)", geonuchoi.com, section 2 GQA): for every sequence s and
// query head h, out = softmax(scale * q K^T) V over the context_lens[s] cached tokens,
// where K/V are reached through the block table and query head h reads K/V head
// h / GROUP.  Blocks are processed one at a time with a running max and running sum, so
// no score vector is ever stored.
//
// GB300 design (decode is HBM-bound: each (block, kv head) tile of 2 KiB of K + 2 KiB of
// V is read once and feeds 4 query heads):
//   * The flattened space of (sequence, kv head, block) tiles is cut into contiguous runs
//     of equal length, one per warp of a persistent grid, so every warp streams the same
//     number of bytes whatever the length mix.  With partition_tokens the runs are at most
//     that long, in equal numbers per warp.
//   * Each warp streams its own run through a private 4-stage ring in shared memory: lane
//     0 issues two tensor-map TMA copies (one 16-row box of each pool, 128-byte swizzle)
//     completing on the stage's mbarrier, and refills a stage as soon as the warp has
//     consumed it.  The block-table entries are fetched 32 at a time, one window ahead.
//     No producer warp, no release barriers, no block-wide synchronisation while
//     streaming.  Before waiting for the previous grid (programmatic dependent launch),
//     a warp with a long run also asks L2 for its next 8 tiles (2 for shorter runs).
//   * The tile arithmetic is a small dense contraction per warp: the GROUP query heads
//     sharing a K/V head against 16 tokens, S = Q K^T ([GROUP x 64] x [64 x 16]) and
//     O += P V ([GROUP x 16] x [16 x 64]).  It runs on the tensor cores as mma.sync
//     m16n8k16 (bf16 in, fp32 accumulate) with the heads as MMA rows (rows past GROUP are
//     zero), K and V fragments loaded by ldmatrix from the swizzled tiles without bank
//     conflicts and P taken from the score accumulators: about 60 instructions per lane
//     and tile, against some 300 for the same arithmetic on the CUDA cores, which left the
//     streaming warps issue-bound.  The quad of lanes of head r keeps its online softmax
//     (running max in log2 units, raised only when a score exceeds it by more than 2^8;
//     running sum of P as rounded to bf16 for the product).
//   * When a piece ends, the quad sums its shares of the running sum and either the final
//     bf16 rows are written (the whole segment in one piece) or an unnormalised (o, max,
//     sum) partial.  The warp that publishes a segment's last piece
//     merges its partials (log-sum-exp weights) inside this kernel, with CTA-scope
//     ordering when all the segment's pieces ran on its CTA; beyond 8192-token contexts
//     or with fixed partitions merge_partials_kernel does it.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kWarps = 12;          // streaming warps per CTA, 3 per SM sub-partition
constexpr int kStagesPerWarp = 4;   // private ring depth: 16 KiB in flight per warp
constexpr int kWindow = 32;         // block-table entries fetched per window
constexpr int kPartialFloats = kHeadDim + 2;  // o[64], max (log2 units), sum
constexpr float kRescaleThreshold = 8.0f;     // log2 units: rescale when max grows > 2^8
constexpr int kMinTilesPerRun = 2;
constexpr int kOneSeqMaxTilesPerWarp = 4;  // a single sequence up to this: one CTA per head
// Before its dependency wait a warp asks L2 for up to kPrefetchTiles tiles past its ring
// (from its first block-table window) when the warps average at least
// kPrefetchMinTilesPerWarp tiles each, kPrefetchTilesShort when they average at least
// kPrefetchShortMinTilesPerWarp, and none when the launch shares the GPU (an SM budget).
constexpr int kPrefetchTiles = 8;
constexpr int kPrefetchMinTilesPerWarp = 48;
constexpr int kPrefetchTilesShort = 2;
constexpr int kPrefetchShortMinTilesPerWarp = 12;
// Longest context whose split segments are merged inside the attention kernel; longer ones
// (many pieces per segment) go to the parallel merge kernel.
constexpr int kFusedMergeMaxContext = 8192;
constexpr int kMaxSeqs = 4096;
constexpr int kMergeThreads = 512;
constexpr int kMergeUnroll = 4;  // partials whose loads one warp has in flight at once
constexpr int kMergeSplitPieces = 16;  // segments with this many pieces merge per query head

struct KParams {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const uint8_t* key_cache;
  const uint8_t* value_cache;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t num_blocks;
  float q_scale;  // scale * log2(e): scores come out in log2 units
  int32_t grid;      // runs of the decomposition (warp w of the grid serves runs
                     // w, w + warps, ...)
  int32_t chunk;     // tiles per run, 0 = balanced split into `grid` runs
  int64_t tile_bound;  // > 0: the host's upper bound of the tile count (partitioned runs)
  int64_t* ws_total;    // total tiles, written by CTA 0
  int32_t* ws_seq_base; // [num_seqs + 1] blocks-per-head prefix, written by CTA 0
  float* partials;      // [runs][2][GROUP][kPartialFloats]
  int32_t* seg_count;   // [num_seqs * Hkv] pieces published per split segment (fused merge);
                        // zero between calls: the merging warp resets its counter
  int32_t fused_merge;  // 1: the last warp to finish a split segment merges it in place
  int32_t prefetch_ok;  // 1: a warp may ask L2 for tiles past its ring before its wait
  const uint8_t* k_new;  // optional [num_seqs][Hkv][64] bf16: token at position L-1 to store
  const uint8_t* v_new;  //   (fused append: stored to its slot and used in attention)
  uint8_t* key_cache_w;    // writable views of the pools (fused append)
  uint8_t* value_cache_w;
  int32_t* status;
  // Mixed batches (the varlen launch): sequence s's query and output row is q_rows[s], and
  // only sequences with exactly one row (q_rows[s+1] - q_rows[s] == 1) are served here; the
  // others are left alone (no tiles, nothing written).  nullptr: row s, every sequence.
  const int32_t* q_rows;
  int32_t num_query_tokens;
};

// Query / output row of sequence s (kRows: the mixed-batch form, a separate instantiation
// so that the plain decode path compiles without it).
template <bool kRows>
__device__ __forceinline__ int64_t row_of(const KParams& p, int s) {
  if (kRows) return p.q_rows[s];
  return s;
}

__device__ __forceinline__ int64_t run_start(int64_t c, int64_t total, int32_t grid,
                                             int32_t chunk) {
  if (chunk > 0) return c * chunk < total ? c * chunk : total;
  return c * total / grid;
}

// Run containing tile x (x < total).  Runs are [run_start(c), run_start(c+1)).
__device__ __forceinline__ int64_t run_of(int64_t x, int64_t total, int32_t grid,
                                          int32_t chunk) {
  if (chunk > 0) return x / chunk;
  return ((x + 1) * grid - 1) / total;
}

// Largest s in [0, num_seqs) with kv * base[s] <= y (y < kv * base[num_seqs]).
__device__ __forceinline__ int find_seq(const int32_t* base, int num_seqs, int64_t y, int kv) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(base[mid]) * kv <= y) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct Piece {
  int s, g, b0, b1, nb;
};

__device__ __forceinline__ Piece piece_at(const int32_t* base, int num_seqs, int kv, int64_t y,
                                          int64_t run_end) {
  Piece pc;
  pc.s = find_seq(base, num_seqs, y, kv);
  pc.nb = base[pc.s + 1] - base[pc.s];
  const int64_t off = y - static_cast<int64_t>(base[pc.s]) * kv;
  pc.g = static_cast<int>(off / pc.nb);
  pc.b0 = static_cast<int>(off % pc.nb);
  const int64_t left = run_end - y;
  pc.b1 = (pc.nb - pc.b0 <= left) ? pc.nb : pc.b0 + static_cast<int>(left);
  return pc;
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int c0, int c1,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Tiles arrive through tensor-map copies with the 128-byte swizzle: the 16-byte chunk c of
// row t (token t, dims 8c .. 8c + 7) sits at t * 128 + ((c ^ (t & 7)) * 16) of its 2 KiB
// stage half, so the eight rows an ldmatrix phase reads fall on eight distinct bank groups.
__device__ __forceinline__ uint32_t swz(int t, int c) {
  return static_cast<uint32_t>(t * kRowBytes + ((c ^ (t & 7)) << 4));
}

// Lane layout of a streaming warp for the tensor-core tile math (mma.sync m16n8k16, bf16
// in, fp32 accumulate): r = lane / 4 is the MMA row (query head r of the group; rows past
// the group and rows 8-15 are zero padding) and q = lane % 4.  S = Q K^T over one 16-token
// tile is two n-tiles of 8 tokens and four k-steps of 16 dims; O += P V takes P straight
// from the score accumulators (tokens 2q, 2q+1, 2q+8, 2q+9 of row r) and V through
// transposing ldmatrix loads; the accumulators of n-tile j hold dims 8j + 2q, 8j + 2q + 1
// of head r.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                          uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// bf16 pair {lo = x, hi = y}
__device__ __forceinline__ uint32_t pack_bf16x2(float x, float y) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// One 16-token tile pair held in shared memory (swizzled).  The quad of row r keeps the
// online-softmax state of head r: m, the running reference maximum in log2 units (raised
// only when a score exceeds it by more than 2^8; the same in the quad's four lanes), and l,
// this lane's share of the running sum of the probabilities as rounded for the P V product.
template <bool TAIL>
__device__ __forceinline__ void attend_tile(uint32_t kt, uint32_t vt, int lane, int q,
                                            int valid_tokens, float q_scale,
                                            const uint32_t (&qa0)[4], const uint32_t (&qa2)[4],
                                            float& m, float& l, float (&o)[8][4]) {
  // K: matrix (n-tile j, chunk c) = tokens 8j .. 8j+7, dims 8c .. 8c+7; an x4 load of
  // chunks 4h .. 4h+3 gives b0/b1 of k-steps 2h and 2h+1.
  const int lrow = lane & 7, lmat = lane >> 3;
  uint32_t k00[4], k01[4], k10[4], k11[4];
  ldsm_x4(kt + swz(lrow, lmat), k00);          // n-tile 0, chunks 0..3
  ldsm_x4(kt + swz(lrow, 4 + lmat), k01);      // n-tile 0, chunks 4..7
  ldsm_x4(kt + swz(8 + lrow, lmat), k10);      // n-tile 1, chunks 0..3
  ldsm_x4(kt + swz(8 + lrow, 4 + lmat), k11);  // n-tile 1, chunks 4..7
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  mma_16816(s0, qa0[0], qa2[0], k00[0], k00[1]);
  mma_16816(s1, qa0[0], qa2[0], k10[0], k10[1]);
  mma_16816(s0, qa0[1], qa2[1], k00[2], k00[3]);
  mma_16816(s1, qa0[1], qa2[1], k10[2], k10[3]);
  mma_16816(s0, qa0[2], qa2[2], k01[0], k01[1]);
  mma_16816(s1, qa0[2], qa2[2], k11[0], k11[1]);
  mma_16816(s0, qa0[3], qa2[3], k01[2], k01[3]);
  mma_16816(s1, qa0[3], qa2[3], k11[2], k11[3]);
  // V: matrix (token half kb, n-tile j) = tokens 8kb .. 8kb+7, dims 8j .. 8j+7, loaded
  // transposed: an x4 load gives b0/b1 of n-tiles j and j+1.  Issued before the softmax so
  // that their latency overlaps it.
  uint32_t v[4][4];
#pragma unroll
  for (int jp = 0; jp < 4; ++jp)
    ldsm_x4_trans(vt + swz(8 * (lmat & 1) + lrow, 2 * jp + (lmat >> 1)), v[jp]);
  float x[4] = {s0[0] * q_scale, s0[1] * q_scale, s1[0] * q_scale, s1[1] * q_scale};
  uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
  if (TAIL) {
    const int t0 = 2 * q;
    if (t0 >= valid_tokens) x[0] = -INFINITY;
    if (t0 + 1 >= valid_tokens) x[1] = -INFINITY;
    if (t0 + 8 >= valid_tokens) x[2] = -INFINITY;
    if (t0 + 9 >= valid_tokens) x[3] = -INFINITY;
    // rows past the context may hold anything (NaN included): P is 0 there, V must be too
    vm0 = (t0 < valid_tokens ? 0x0000ffffu : 0u) | (t0 + 1 < valid_tokens ? 0xffff0000u : 0u);
    vm1 = (t0 + 8 < valid_tokens ? 0x0000ffffu : 0u) | (t0 + 9 < valid_tokens ? 0xffff0000u : 0u);
  }
  float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
  mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
  const bool grow = mt - m > kRescaleThreshold;  // first tile: m = -inf
  if (__any_sync(0xffffffffu, grow)) {
    const float alpha = grow ? fast_exp2(m - mt) : 1.f;
    if (grow) m = mt;
    l *= alpha;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j][0] *= alpha;
      o[j][1] *= alpha;
    }
  }
  const uint32_t pa0 = pack_bf16x2(fast_exp2(x[0] - m), fast_exp2(x[1] - m));
  const uint32_t pa2 = pack_bf16x2(fast_exp2(x[2] - m), fast_exp2(x[3] - m));
  {
    const float2 f0 = bf16x2_to_float2(pa0), f2 = bf16x2_to_float2(pa2);
    l += (f0.x + f0.y) + (f2.x + f2.y);
  }
#pragma unroll
  for (int jp = 0; jp < 4; ++jp) {
    mma_16816(o[2 * jp], pa0, pa2, v[jp][0] & vm0, v[jp][1] & vm1);
    mma_16816(o[2 * jp + 1], pa0, pa2, v[jp][2] & vm0, v[jp][3] & vm1);
  }
}

template <int GROUP>
constexpr size_t decode_smem_fixed() {
  return static_cast<size_t>(kWarps) *
         (kStagesPerWarp * 2 * kTileBytes          // private K+V rings
          + kStagesPerWarp * sizeof(uint64_t)      // full barriers
          + kStagesPerWarp * sizeof(int32_t));     // tile id held by each stage
}

// Block-table window: lane j holds the tile (phys_block * Hkv + kv_head) of the j-th of
// `n` consecutive tiles of one run, or -1 for an invalid block id.
struct Window {
  int32_t tile;  // raw block id until resolved (see resolve_window), then the tile or -1
  int32_t g;
  int n;
};

// Pieces of segment [x0, x1) (one (sequence, kv head)): the non-empty runs it touches.  The
// first piece sits in slot 0 of its run when the segment starts the run, else in slot 1;
// every later piece starts its run (slot 0).
struct SegmentPieces {
  int64_t c_first, c_last;
  int first_slot;
};

__device__ __forceinline__ SegmentPieces segment_pieces(int64_t x0, int64_t x1, int64_t total,
                                                        int32_t runs, int32_t chunk) {
  SegmentPieces sp;
  sp.c_first = run_of(x0, total, runs, chunk);
  sp.c_last = run_of(x1 - 1, total, runs, chunk);
  sp.first_slot = x0 == run_start(sp.c_first, total, runs, chunk) ? 0 : 1;
  return sp;
}

// Number of pieces of a segment, and the run holding piece k (balanced splits only, which
// is the only mode that merges inside the attention kernel).  With at least one tile per
// run (total >= runs) every run is non-empty and piece k lies in run c_first + k; otherwise
// every non-empty run holds exactly one tile and piece k is the run of tile x0 + k.
__device__ __forceinline__ int segment_piece_count(const SegmentPieces& sp, int64_t x0, int64_t x1,
                                                   int64_t total, int32_t runs) {
  return total >= runs ? static_cast<int>(sp.c_last - sp.c_first + 1) : static_cast<int>(x1 - x0);
}
__device__ __forceinline__ int64_t segment_piece_run(const SegmentPieces& sp, int64_t x0, int k,
                                                     int64_t total, int32_t runs, int32_t chunk) {
  return total >= runs ? sp.c_first + k : run_of(x0 + k, total, runs, chunk);
}

// One warp combines all pieces of a split segment (log-sum-exp weights) and writes the bf16
// rows of its GROUP query heads.  Lane k reads piece k's (max, sum), so the pieces' loads
// overlap; chunks of 32 pieces are combined with a running maximum.  Partials were written
// by other warps in this launch, so they are read through L2 (__ldcg), after the caller's
// acquire fence.
constexpr int kFewPieces = 4;  // segments of up to this many pieces merge in one load round

// Partials written by warps of this CTA (published with CTA-scope ordering) are read with
// plain loads; partials from other SMs through L2.
template <bool kLocal>
__device__ __forceinline__ float ld_partial(const float* a) {
  return kLocal ? *a : __ldcg(a);
}
template <bool kLocal>
__device__ __forceinline__ float2 ld_partial2(const float2* a) {
  return kLocal ? *a : __ldcg(a);
}

template <int GROUP, bool kLocal, bool kRows>
__device__ void merge_segment_in_warp(const KParams& p, const SegmentPieces& sp, int64_t x0,
                                      int64_t x1, int64_t total, int s, int g, int lane) {
  const int n = segment_piece_count(sp, x0, x1, total, p.grid);
  if (n <= kFewPieces) {
    // Few pieces (the usual case): every lane loads the (max, sum) of all pieces and its
    // own output slice of each, all in one round of loads, and combines them in registers.
    float mk[kFewPieces][GROUP], lk[kFewPieces][GROUP];
    float2 vk[kFewPieces][GROUP];
#pragma unroll
    for (int k = 0; k < kFewPieces; ++k) {
      if (k < n) {
        const int64_t c = segment_piece_run(sp, x0, k, total, p.grid, p.chunk);
        const int slot = k == 0 ? sp.first_slot : 0;
        const float* rec = p.partials + (c * 2 + slot) * GROUP * kPartialFloats;
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
          mk[k][h] = ld_partial<kLocal>(rec + h * kPartialFloats + kHeadDim);
          lk[k][h] = ld_partial<kLocal>(rec + h * kPartialFloats + kHeadDim + 1);
          vk[k][h] = ld_partial2<kLocal>(reinterpret_cast<const float2*>(rec + h * kPartialFloats) + lane);
        }
      } else {
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
          mk[k][h] = -INFINITY;
          lk[k][h] = 0.f;
          vk[k][h] = make_float2(0.f, 0.f);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
      float mh = mk[0][h];
#pragma unroll
      for (int k = 1; k < kFewPieces; ++k) mh = fmaxf(mh, mk[k][h]);
      float lh = 0.f;
      float2 ah = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kFewPieces; ++k) {
        const float wgt = k < n ? fast_exp2(mk[k][h] - mh) : 0.f;
        lh += wgt * lk[k][h];
        ah.x += wgt * vk[k][h].x;
        ah.y += wgt * vk[k][h].y;
      }
      const float inv = 1.f / lh;
      __nv_bfloat16* out =
          p.out + (row_of<kRows>(p, s) * p.num_q_heads + g * GROUP + h) * kHeadDim;
      reinterpret_cast<__nv_bfloat162*>(out)[lane] = __floats2bfloat162_rn(ah.x * inv, ah.y * inv);
    }
    return;
  }
  float M[GROUP], L[GROUP];
  float2 acc[GROUP];
#pragma unroll
  for (int h = 0; h < GROUP; ++h) {
    M[h] = -INFINITY;
    L[h] = 0.f;
    acc[h] = make_float2(0.f, 0.f);
  }
  for (int base = 0; base < n; base += 32) {
    const int k = base + lane;
    const bool valid = k < n;
    const float* rec = p.partials;
    if (valid) {
      const int64_t c = segment_piece_run(sp, x0, k, total, p.grid, p.chunk);
      const int slot = k == 0 ? sp.first_slot : 0;
      rec = p.partials + (c * 2 + slot) * GROUP * kPartialFloats;
    }
    // every head's (max, sum) of piece k, all loads in flight together
    float mk[GROUP], lk[GROUP], wk[GROUP];
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
      mk[h] = valid ? ld_partial<kLocal>(rec + h * kPartialFloats + kHeadDim) : -INFINITY;
      lk[h] = valid ? ld_partial<kLocal>(rec + h * kPartialFloats + kHeadDim + 1) : 0.f;
    }
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
      float cm = mk[h];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
      const float nm = fmaxf(M[h], cm);
      const float keep = M[h] == -INFINITY ? 0.f : fast_exp2(M[h] - nm);
      wk[h] = valid ? fast_exp2(mk[h] - nm) : 0.f;
      float lw = wk[h] * lk[h];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
      L[h] = L[h] * keep + lw;
      acc[h].x *= keep;
      acc[h].y *= keep;
      M[h] = nm;
    }
    // output slices: 4 pieces x GROUP heads of loads in flight per round
    const int cnt = min(32, n - base);
    for (int j0 = 0; j0 < cnt; j0 += 4) {
      float2 v[4][GROUP];
      float w[4][GROUP];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u < cnt ? j0 + u : j0;  // clamp; weight zeroed below
        const float* rj = reinterpret_cast<const float*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(rec), j));
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
          w[u][h] = __shfl_sync(0xffffffffu, wk[h], j);
          if (j0 + u >= cnt) w[u][h] = 0.f;
          v[u][h] = ld_partial2<kLocal>(reinterpret_cast<const float2*>(rj + h * kPartialFloats) + lane);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
          acc[h].x += w[u][h] * v[u][h].x;
          acc[h].y += w[u][h] * v[u][h].y;
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < GROUP; ++h) {
    const float inv = 1.f / L[h];
    __nv_bfloat16* out =
        p.out + (row_of<kRows>(p, s) * p.num_q_heads + g * GROUP + h) * kHeadDim;
    reinterpret_cast<__nv_bfloat162*>(out)[lane] =
        __floats2bfloat162_rn(acc[h].x * inv, acc[h].y * inv);
  }
}

template <int GROUP, bool kRows>
__global__ void __launch_bounds__(kWarps * 32, 1)
paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const KParams p) {
  constexpr int kThreads = kWarps * 32;
  // A launch that follows in the stream with programmatic dependent launch enabled may
  // start as soon as SMs free up; it waits for this grid before it reads what this grid
  // writes (griddepcontrol.wait below).  No effect on launches without that attribute.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(1024) uint8_t smem[];  // 128-byte swizzle atoms need 1 KiB
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.num_seqs;
  const int KV = p.num_kv_heads;

  uint8_t* ring = smem + warp * (kStagesPerWarp * 2 * kTileBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * kStagesPerWarp * 2 * kTileBytes);
  uint64_t* full_bar = bars + warp * kStagesPerWarp;
  int32_t* stage_tile = reinterpret_cast<int32_t*>(bars + kWarps * kStagesPerWarp) +
                        warp * kStagesPerWarp;
  int32_t* seq_base = reinterpret_cast<int32_t*>(bars + kWarps * kStagesPerWarp) +
                      kWarps * kStagesPerWarp;
  __shared__ int64_t warp_sums[kWarps];
  // piece counters of split segments whose pieces all run on this CTA, by the segment's
  // first run modulo kWarps (two such segments never share a first run)
  __shared__ int cta_seg_count[kWarps];
  if (tid < kWarps) cta_seg_count[tid] = 0;
  if ((smem_addr(smem) & 1023u) != 0) {  // never issue swizzled copies to a misaligned ring
    if (tid == 0 && blockIdx.x == 0) flag_error(p.status, PA_DEVFLAG_LAYOUT);
    return;
  }

  if (lane == 0) {
    for (int i = 0; i < kStagesPerWarp; ++i) mbar_init(&full_bar[i], 1);
    fence_barrier_init();
  }

  // Query rows (and, with the fused append, the new K/V rows) are read when a piece starts,
  // often in the middle of a warp's stream: bring all of them into L2 now, one 128-byte row
  // per thread of the grid.
  {
    const int64_t q_rows = kRows ? 0 : static_cast<int64_t>(S) * p.num_q_heads;
    const int64_t kv_rows = p.k_new != nullptr ? static_cast<int64_t>(S) * KV : 0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + tid; i < q_rows + 2 * kv_rows;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
      const uint8_t* row =
          i < q_rows ? reinterpret_cast<const uint8_t*>(p.q) + i * kRowBytes
          : i < q_rows + kv_rows ? p.k_new + (i - q_rows) * kRowBytes
                                 : p.v_new + (i - q_rows - kv_rows) * kRowBytes;
      prefetch_l2(row);
    }
  }

  // ---- per-sequence block counts and their exclusive prefix (the tile index space) ----
  for (int i = tid; i < S; i += kThreads) {
    const int32_t L = p.context_lens[i];
    int32_t nb = 0;
    bool serve = true;
    if (kRows) {  // mixed batch: decode rows only, the same checks as chunks
      const int32_t r0 = p.q_rows[i];
      const int32_t q_len = p.q_rows[i + 1] - r0;
      serve = q_len == 1;
      if (serve && (r0 < 0 || r0 >= p.num_query_tokens || L < 1)) {
        if (blockIdx.x == 0) flag_error(p.status, PA_DEVFLAG_BAD_CONTEXT);
        serve = false;
      }
    }
    if (!serve) {
    } else if (L < 0 || static_cast<int64_t>(L) > static_cast<int64_t>(p.max_blocks_per_seq) * kBlockSize) {
      if (blockIdx.x == 0) flag_error(p.status, PA_DEVFLAG_BAD_CONTEXT);
    } else {
      nb = (L + kBlockSize - 1) / kBlockSize;
    }
    seq_base[i] = nb;
  }
  __syncthreads();
  {
    const int per = (S + kThreads - 1) / kThreads;
    const int beg = min(tid * per, S);
    const int end = min(beg + per, S);
    int64_t local = 0;
    for (int i = beg; i < end; ++i) local += seq_base[i];
    int64_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int64_t run = incl - local;
    int64_t grand = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) run += warp_sums[w];
      grand += warp_sums[w];
    }
    const bool overflow = grand * KV > 0x7fffffffLL;
    for (int i = beg; i < end; ++i) {
      const int32_t v = seq_base[i];
      seq_base[i] = static_cast<int32_t>(overflow ? 0 : run);
      run += v;
    }
    if (tid == 0) seq_base[S] = static_cast<int32_t>(overflow ? 0 : grand);
    if (overflow && tid == 0 && blockIdx.x == 0) flag_error(p.status, PA_DEVFLAG_BAD_CONTEXT);
  }
  __syncthreads();

  const int64_t total = static_cast<int64_t>(seq_base[S]) * KV;
  // From here on every warp works alone: no block-wide synchronisation below.
  const int64_t total_warps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (gw >= p.grid) return;

  const uint64_t policy = l2_evict_first_policy();
  const int r = lane >> 2;  // MMA row: query head r of the group (padding past GROUP)
  const int q = lane & 3;

  // ---- issue side: the warp's runs, walked one block-table window at a time ----
  int64_t wc_run = gw;
  int64_t wc_y = run_start(gw, total, p.grid, p.chunk);
  int64_t wc_stop = run_start(gw + 1, total, p.grid, p.chunk);
  auto next_window = [&]() -> Window {
    while (wc_y >= wc_stop && wc_run < p.grid) {
      wc_run += total_warps;
      if (wc_run < p.grid) {
        wc_y = run_start(wc_run, total, p.grid, p.chunk);
        wc_stop = run_start(wc_run + 1, total, p.grid, p.chunk);
      }
    }
    Window w;
    w.tile = 0;
    w.g = 0;
    const int64_t left = wc_stop - wc_y;
    w.n = wc_run < p.grid ? static_cast<int>(left < kWindow ? left : kWindow) : 0;
    if (lane < w.n) {
      const int64_t y = wc_y + lane;
      const int s = find_seq(seq_base, S, y, KV);
      const int nb = seq_base[s + 1] - seq_base[s];
      const int off = static_cast<int>(y - static_cast<int64_t>(seq_base[s]) * KV);
      const int g = off / nb;
      const int b = off - g * nb;
      w.tile = __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq + b);
      w.g = g;
    }
    wc_y += w.n;
    return w;
  };
  // The loaded block ids are checked and turned into tiles only when the window is first
  // used, so that the loads of the next window stay in flight meanwhile.
  auto resolve_window = [&](Window& w) {
    const bool bad = lane < w.n && (w.tile < 0 || w.tile >= p.num_blocks);
    w.tile = lane < w.n && !bad ? w.tile * KV + w.g : -1;
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_error(p.status, PA_DEVFLAG_BAD_BLOCK);
  };
  Window cur = next_window();
  Window nxt = next_window();
  resolve_window(cur);
  int cur_i = 0;
  int issued = 0;
  auto issue_one = [&]() {
    if (cur_i >= cur.n) {
      cur = nxt;
      cur_i = 0;
      if (cur.n == 0) return;  // nothing left to issue
      resolve_window(cur);
      nxt = next_window();
    }
    const int32_t t = __shfl_sync(0xffffffffu, cur.tile, cur_i);
    const int st = issued % kStagesPerWarp;
    if (lane == 0) {
      stage_tile[st] = t;  // read back by the fused append
      if (t >= 0) {
        mbar_arrive_expect_tx(&full_bar[st], 2 * kTileBytes);
        uint8_t* dst = ring + st * 2 * kTileBytes;
        // one 16-row box per pool: rows t*16 .. t*16+15 of the [rows][64] view, swizzled
        tma_load_2d_hint(dst, &tmap_k, 0, t * kBlockSize, &full_bar[st], policy);
        tma_load_2d_hint(dst + kTileBytes, &tmap_v, 0, t * kBlockSize, &full_bar[st], policy);
      } else {
        mbar_arrive(&full_bar[st]);  // invalid block: release the stage with stale data
      }
    }
    ++issued;
    ++cur_i;
  };
  for (int i = 0; i < kStagesPerWarp; ++i) issue_one();
  // The next tiles of the first window, past the ring, are requested into L2 now: under
  // programmatic dependent launch the wait below lasts until the previous grid's slowest
  // CTAs end, and with long runs per warp the extra requests keep DRAM busy meanwhile
  // (and at the start of a launch).  Lane i holds entry i of the window; entries before
  // cur_i are in the ring already.
  const int64_t busy_warps = p.grid < total_warps ? p.grid : total_warps;
  const int pf = !p.prefetch_ok                                        ? 0
                 : total >= kPrefetchMinTilesPerWarp * busy_warps      ? kPrefetchTiles
                 : total >= kPrefetchShortMinTilesPerWarp * busy_warps ? kPrefetchTilesShort
                                                                       : 0;
  if (pf > 0 && lane >= cur_i && lane < cur.n && lane < cur_i + pf && cur.tile >= 0) {
    const int64_t off = static_cast<int64_t>(cur.tile) * kTileBytes;
    bulk_prefetch_l2(p.key_cache + off, kTileBytes, policy);  // evict-first, as the loads
    bulk_prefetch_l2(p.value_cache + off, kTileBytes, policy);
  }

  // Everything above reads only block_tables, context_lens (q_rows) and K/V tiles.  Under
  // programmatic dependent launch the previous kernel in the stream may still be running
  // here; wait for it (and its memory) before reading queries or new K/V rows and before
  // writing outputs or the workspace.  Without that launch attribute this returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (blockIdx.x == 0 && warp == 0) {  // warp 0 of CTA 0 always runs (grid >= 1 run)
    for (int i = lane; i <= S; i += 32) p.ws_seq_base[i] = seq_base[i];
    if (lane == 0) {
      *p.ws_total = total;
      if ((p.chunk > 0 && static_cast<int64_t>(p.grid) * p.chunk < total) ||
          (p.tile_bound > 0 && total > p.tile_bound))
        flag_error(p.status, PA_DEVFLAG_BAD_CONTEXT);  // contexts beyond max_context_len
    }
    if (p.fused_merge && !kRows) {
      // empty contexts: zero rows (no tile writes them)
      const int row_elems = p.num_q_heads * kHeadDim;
      for (int s0 = 0; s0 < S; ++s0) {
        if (seq_base[s0 + 1] != seq_base[s0]) continue;
        __nv_bfloat16* out = p.out + static_cast<int64_t>(s0) * row_elems;
        for (int e = lane; e < row_elems; e += 32) out[e] = __float2bfloat16_rn(0.f);
      }
    }
  }

  // ---- consume side: same runs, piece by piece ----
  int waited = 0;  // tiles whose data this warp has waited for (stage = waited % stages)
  bool ok = true;
  for (int64_t run = gw; run < p.grid; run += total_warps) {
  const int64_t start = run_start(run, total, p.grid, p.chunk);
  const int64_t stop = run_start(run + 1, total, p.grid, p.chunk);
  for (int64_t y = start; y < stop;) {
    const Piece pc = piece_at(seq_base, S, KV, y, stop);
    const int32_t L = p.context_lens[pc.s];
    const bool whole = pc.b0 == 0 && pc.b1 == pc.nb;
    const bool first_piece = y == start;
    const int ntiles = pc.b1 - pc.b0;

    uint32_t qa0[4] = {0u, 0u, 0u, 0u}, qa2[4] = {0u, 0u, 0u, 0u};
    if (r < GROUP) {
      const __nv_bfloat16* qrow =
          p.q + (row_of<kRows>(p, pc.s) * p.num_q_heads + pc.g * GROUP + r) * kHeadDim;
      const uint32_t* qw = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {  // dims 16ks + 2q (+1) and 16ks + 8 + 2q (+1)
        qa0[ks] = __ldg(qw + 8 * ks + q);
        qa2[ks] = __ldg(qw + 8 * ks + 4 + q);
      }
    }
    // Fused append: this piece holds the (sequence, kv head)'s last tile, whose row
    // (L - 1) % 16 is the new token.  Lanes 0-7 carry its K chunks, 8-15 its V chunks.
    const bool append_here = p.k_new != nullptr && pc.b1 == pc.nb && lane < 16;
    uint4 new_row = make_uint4(0, 0, 0, 0);
    if (append_here) {
      const uint8_t* src = (lane < 8 ? p.k_new : p.v_new) +
                           (static_cast<int64_t>(pc.s) * KV + pc.g) * kRowBytes + (lane & 7) * 16;
      new_row = ldg_nc128(src);
    }
    float m = -INFINITY, l = 0.f;
    float o[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

    for (int k = 0; k < ntiles && ok; ++k) {
      const int st = waited % kStagesPerWarp;
      const uint32_t phase = static_cast<uint32_t>((waited / kStagesPerWarp) & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[st], phase))) {
        if (lane == 0) flag_error(p.status, PA_DEVFLAG_TIMEOUT);
        ok = false;
        break;
      }
      ++waited;
      uint8_t* kt = ring + st * 2 * kTileBytes;
      uint8_t* vt = kt + kTileBytes;
      const int valid = L - (pc.b0 + k) * kBlockSize;
      if (p.k_new != nullptr && pc.b0 + k == pc.nb - 1) {
        // the new token: into the tile before it is read, and into its slot in the pools
        if (append_here) {
          const int nrow = (L - 1) % kBlockSize;
          const int off = nrow * kRowBytes + (lane & 7) * 16;  // place in the pools
          uint8_t* tile = lane < 8 ? kt : vt;
          *reinterpret_cast<uint4*>(tile + swz(nrow, lane & 7)) = new_row;  // swizzled stage
          const int32_t t = stage_tile[st];
          if (t >= 0) {
            uint8_t* pool = lane < 8 ? p.key_cache_w : p.value_cache_w;
            *reinterpret_cast<uint4*>(pool + static_cast<size_t>(t) * kTileBytes + off) = new_row;
          }
          // This stage is refilled by a TMA copy (async proxy) after the tile is consumed.
          // A generic-proxy write followed by an async-proxy write to the same shared memory
          // is ordered only through a proxy fence: without it the new row could land after
          // the refill and corrupt the next tile.  (Plain reads need no fence: their values
          // have been consumed before the warp barrier that precedes the refill.)
          fence_proxy_async_smem();
        }
        __syncwarp();
      }
      if (valid >= kBlockSize) {
        attend_tile<false>(smem_addr(kt), smem_addr(vt), lane, q, kBlockSize, p.q_scale, qa0, qa2,
                           m, l, o);
      } else {
        attend_tile<true>(smem_addr(kt), smem_addr(vt), lane, q, valid, p.q_scale, qa0, qa2, m,
                          l, o);
      }
      // Every lane's reads of this stage have completed (their values fed the arithmetic
      // above); the warp barrier orders them before lane 0 issues the refill into the same
      // buffer, as a consumer's release orders its reads before a producer's next copy.
      __syncwarp();
      issue_one();
    }

    // ---- the quad of row r holds head r: sum its four shares of l ----
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (r < GROUP) {
      if (whole) {
        const float inv = 1.f / l;
        const int64_t row = row_of<kRows>(p, pc.s) * p.num_q_heads + pc.g * GROUP + r;
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + row * kHeadDim);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[4 * j + q] = pack_bf16x2(o[j][0] * inv, o[j][1] * inv);
      } else {
        const int slot = first_piece ? 0 : 1;
        float* dst = p.partials + ((run * 2 + slot) * GROUP + r) * kPartialFloats;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float2*>(dst + 8 * j + 2 * q) = make_float2(o[j][0], o[j][1]);
        if (q == 0) {
          dst[kHeadDim] = m;
          dst[kHeadDim + 1] = l;
        }
      }
    }
    if (!whole && p.fused_merge) {
      // Publish this piece; the warp that publishes the segment's last piece merges it.
      // When every piece of the segment runs on this CTA (one round of runs, all its runs
      // among this CTA's kWarps), publishing needs only CTA-scope ordering and a shared
      // counter; otherwise device-scope fences and the workspace counter.
      const int64_t x0 = static_cast<int64_t>(seq_base[pc.s]) * KV + static_cast<int64_t>(pc.g) * pc.nb;
      const SegmentPieces sp = segment_pieces(x0, x0 + pc.nb, total, p.grid, p.chunk);
      const bool local = p.grid <= total_warps && sp.c_first / kWarps == sp.c_last / kWarps;
      int last = 0;
      if (local) {
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          const int n = segment_piece_count(sp, x0, x0 + pc.nb, total, p.grid);
          last = atomicAdd(&cta_seg_count[sp.c_first % kWarps], 1) == n - 1;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
          __threadfence_block();  // acquire the other pieces' partials
          merge_segment_in_warp<GROUP, true, kRows>(p, sp, x0, x0 + pc.nb, total, pc.s, pc.g, lane);
          if (lane == 0) cta_seg_count[sp.c_first % kWarps] = 0;
        }
      } else {
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          const int n = segment_piece_count(sp, x0, x0 + pc.nb, total, p.grid);
          last = atomicAdd(&p.seg_count[pc.s * KV + pc.g], 1) == n - 1;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
          __threadfence();  // acquire the other pieces' partials
          merge_segment_in_warp<GROUP, false, kRows>(p, sp, x0, x0 + pc.nb, total, pc.s, pc.g, lane);
          if (lane == 0) p.seg_count[pc.s * KV + pc.g] = 0;  // ready for the next call
        }
      }
    }
    y += ntiles;
  }
  }
  // After a timeout, leave no copy in flight into this warp's ring (bounded waits).
  if (!ok && lane == 0) {
    for (int t = waited; t < issued; ++t) {
      if (!mbar_wait(&full_bar[t % kStagesPerWarp],
                     static_cast<uint32_t>((t / kStagesPerWarp) & 1))) break;
    }
  }
}

// Combines the partials of every (sequence, kv head) whose tiles were split across CTAs,
// and writes zero rows for empty contexts.  One CTA per (sequence, kv head, HPC of the
// head's GROUP query heads): HPC = GROUP when segments have few pieces, 1 when they have
// many (long contexts), so that GROUP times as many CTAs share the loads.  Each warp folds
// its partials into a running (maximum, sum, o) per query head, rescaling by the
// log-sum-exp weights as the maximum grows, with U partials' loads in flight per round;
// the warps' states are then combined the same way.
template <int GROUP, int HPC, bool kRows>
__global__ void __launch_bounds__(kMergeThreads)
merge_partials_kernel(const KParams p) {
  constexpr int kWarps = kMergeThreads / 32;
  constexpr int kSplit = GROUP / HPC;
  constexpr int U = HPC == 1 ? 2 * kMergeUnroll : kMergeUnroll;
  __shared__ float red_m[kWarps][HPC];
  __shared__ float red_l[kWarps][HPC];
  __shared__ float red_o[kWarps][HPC][kHeadDim];
  const int g = blockIdx.x / kSplit;
  const int h0 = (blockIdx.x % kSplit) * HPC;
  const int s = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int KV = p.num_kv_heads;
  __nv_bfloat16* out =
      p.out + (row_of<kRows>(p, s) * p.num_q_heads + g * GROUP + h0) * kHeadDim;
  const int32_t base = p.ws_seq_base[s];
  const int nb = p.ws_seq_base[s + 1] - base;
  if (nb == 0) {
    // an empty context gives a zero row; in a mixed batch nb == 0 means the sequence is not
    // a decode row (or was flagged), and its row is left alone
    if (!kRows)
      for (int e = tid; e < HPC * kHeadDim; e += kMergeThreads) out[e] = __float2bfloat16_rn(0.f);
    return;
  }
  const int64_t total = *p.ws_total;
  const int64_t x0 = static_cast<int64_t>(base) * KV + static_cast<int64_t>(g) * nb;
  const int64_t x1 = x0 + nb;
  const int64_t c_first = run_of(x0, total, p.grid, p.chunk);
  const int64_t c_last = run_of(x1 - 1, total, p.grid, p.chunk);
  if (c_last >= p.grid) {  // tiles beyond the grid (contexts above max_context_len)
    if (tid == 0) flag_error(p.status, PA_DEVFLAG_BAD_CONTEXT);
    return;
  }
  if (c_first == c_last) return;  // written directly by the attention kernel
  const int n = static_cast<int>(c_last - c_first + 1);
  const int first_slot = x0 == run_start(c_first, total, p.grid, p.chunk) ? 0 : 1;

  auto record = [&](int k, int h) -> const float* {
    const int64_t c = c_first + k;
    const int slot = k == 0 ? first_slot : 0;
    return p.partials + ((c * 2 + slot) * GROUP + h0 + h) * kPartialFloats;
  };
  // With at least one tile per run (the usual case) no run is empty and the test is skipped.
  const bool maybe_empty = total < p.grid;
  auto empty_run = [&](int k) -> bool {
    if (!maybe_empty) return false;
    const int64_t c = c_first + k;
    return run_start(c, total, p.grid, p.chunk) == run_start(c + 1, total, p.grid, p.chunk);
  };

  float M[HPC], L[HPC];
  float2 A[HPC];
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    M[h] = -INFINITY;
    L[h] = 0.f;
    A[h] = make_float2(0.f, 0.f);
  }
  // Each warp takes U partials per round and issues all their loads before combining them,
  // so a round costs one memory latency.
  for (int k0 = warp * U; k0 < n; k0 += kWarps * U) {
    float mk[U][HPC], lk[U][HPC];
    float2 vk[U][HPC];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = k0 + u;
      const bool use = k < n && !empty_run(k);
#pragma unroll
      for (int h = 0; h < HPC; ++h) {
        if (use) {
          const float* r = record(k, h);
          mk[u][h] = r[kHeadDim];
          lk[u][h] = r[kHeadDim + 1];
          vk[u][h] = *reinterpret_cast<const float2*>(r + 2 * lane);
        } else {
          mk[u][h] = -INFINITY;
          lk[u][h] = 0.f;
          vk[u][h] = make_float2(0.f, 0.f);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
      float mu = mk[0][h];
#pragma unroll
      for (int u = 1; u < U; ++u) mu = fmaxf(mu, mk[u][h]);
      const float nm = fmaxf(M[h], mu);
      if (nm == -INFINITY) continue;  // nothing of this head loaded yet
      const float keep = M[h] == -INFINITY ? 0.f : fast_exp2(M[h] - nm);
      L[h] *= keep;
      A[h].x *= keep;
      A[h].y *= keep;
      M[h] = nm;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float wgt = mk[u][h] == -INFINITY ? 0.f : fast_exp2(mk[u][h] - nm);
        L[h] += wgt * lk[u][h];
        A[h].x += wgt * vk[u][h].x;
        A[h].y += wgt * vk[u][h].y;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    red_o[warp][h][2 * lane] = A[h].x;
    red_o[warp][h][2 * lane + 1] = A[h].y;
    if (lane == 0) {
      red_m[warp][h] = M[h];
      red_l[warp][h] = L[h];
    }
  }
  __syncthreads();
  for (int e = tid; e < HPC * kHeadDim; e += kMergeThreads) {
    const int h = e / kHeadDim;
    const int d = e % kHeadDim;
    float gm = -INFINITY;
    for (int w = 0; w < kWarps; ++w) gm = fmaxf(gm, red_m[w][h]);
    float o = 0.f, lsum = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      if (red_m[w][h] == -INFINITY) continue;  // a warp without partials
      const float wgt = fast_exp2(red_m[w][h] - gm);
      o += wgt * red_o[w][h][d];
      lsum += wgt * red_l[w][h];
    }
    out[e] = __float2bfloat16_rn(o / lsum);
  }
}

template <int GROUP>
size_t smem_bytes(int num_seqs) {
  return decode_smem_fixed<GROUP>() + sizeof(int32_t) * (num_seqs + 1);
}

template <int GROUP, bool kRows>
cudaError_t prepare_one() {
  static bool done = false;  // benign race: the attribute call is idempotent
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<GROUP, kRows>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_bytes<GROUP>(kMaxSeqs)));
  if (e == cudaSuccess)  // the ring needs the full shared-memory carveout
    e = cudaFuncSetAttribute(paged_decode_kernel<GROUP, kRows>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done = true;
  return e;
}

template <int GROUP>
cudaError_t prepare_kernel() {
  cudaError_t e = prepare_one<GROUP, false>();
  return e == cudaSuccess ? prepare_one<GROUP, true>() : e;
}

// Both instantiations have the same resources; the plan sizes the grid from the plain one.
template <int GROUP>
cudaError_t occupancy(int num_seqs, int* ctas_per_sm) {
  cudaError_t e = prepare_kernel<GROUP>();
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      ctas_per_sm, paged_decode_kernel<GROUP, false>, kWarps * 32,
      smem_bytes<GROUP>(num_seqs));
}

template <int GROUP>
cudaError_t launch(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
  cudaError_t e = prepare_kernel<GROUP>();
  if (e != cudaSuccess) return e;
  KParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.key_cache = static_cast<const uint8_t*>(a.key_cache);
  p.value_cache = static_cast<const uint8_t*>(a.value_cache);
  p.block_tables = a.block_tables;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.context_lens = a.context_lens;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.q_scale = a.scale * 1.4426950408889634f;
  p.grid = plan.runs;
  p.chunk = plan.chunk;
  p.tile_bound = plan.tile_bound;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.ws_total = reinterpret_cast<int64_t*>(ws);
  p.ws_seq_base = reinterpret_cast<int32_t*>(ws + 16);
  p.seg_count = reinterpret_cast<int32_t*>(ws + plan.ws_count_offset);
  p.partials = reinterpret_cast<float*>(ws + plan.ws_meta_bytes);
  p.fused_merge = plan.fused_merge ? 1 : 0;
  p.prefetch_ok = plan.prefetch_ok ? 1 : 0;
  p.k_new = static_cast<const uint8_t*>(a.k_new);
  p.v_new = static_cast<const uint8_t*>(a.v_new);
  p.key_cache_w = static_cast<uint8_t*>(const_cast<void*>(a.key_cache));
  p.value_cache_w = static_cast<uint8_t*>(const_cast<void*>(a.value_cache));
  p.status = a.status;
  p.q_rows = a.q_rows;
  p.num_query_tokens = a.num_query_tokens;
  CUtensorMap tk, tv;
  const uint64_t pool_rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  if (pool_rows >= (1ull << 31) || !encode_pool_rows(&tk, a.key_cache, pool_rows, kBlockSize) ||
      !encode_pool_rows(&tv, a.value_cache, pool_rows, kBlockSize))
    return cudaErrorInvalidValue;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.overlap_previous ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = a.q_rows != nullptr ? cudaLaunchKernelEx(&cfg, paged_decode_kernel<GROUP, true>, tk, tv, p)
                            : cudaLaunchKernelEx(&cfg, paged_decode_kernel<GROUP, false>, tk, tv, p);
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  if (e != cudaSuccess || plan.fused_merge) return e;
  if (plan.merge_split_heads && GROUP > 1) {  // one CTA per query head
    const dim3 mgrid(a.num_kv_heads * GROUP, a.num_seqs);
    if (a.q_rows != nullptr)
      merge_partials_kernel<GROUP, 1, true><<<mgrid, kMergeThreads, 0, stream>>>(p);
    else
      merge_partials_kernel<GROUP, 1, false><<<mgrid, kMergeThreads, 0, stream>>>(p);
  } else {  // one CTA per kv head
    const dim3 mgrid(a.num_kv_heads, a.num_seqs);
    if (a.q_rows != nullptr)
      merge_partials_kernel<GROUP, GROUP, true><<<mgrid, kMergeThreads, 0, stream>>>(p);
    else
      merge_partials_kernel<GROUP, GROUP, false><<<mgrid, kMergeThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t plan_decode(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                        int32_t max_context_len, int32_t partition_tokens, DecodePlan* plan,
                        int32_t max_sms) {
  const int group = num_q_heads / num_kv_heads;
  plan->group = group;
  int ctas_per_sm = 0;
  cudaError_t e;
  switch (group) {
    case 1: e = occupancy<1>(num_seqs, &ctas_per_sm); plan->smem_bytes = smem_bytes<1>(num_seqs); break;
    case 2: e = occupancy<2>(num_seqs, &ctas_per_sm); plan->smem_bytes = smem_bytes<2>(num_seqs); break;
    case 4: e = occupancy<4>(num_seqs, &ctas_per_sm); plan->smem_bytes = smem_bytes<4>(num_seqs); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (ctas_per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t blocks_max = (static_cast<int64_t>(max_context_len) + kBlockSize - 1) / kBlockSize;
  const int64_t tiles_upper = static_cast<int64_t>(num_seqs) * num_kv_heads * blocks_max;
  // max_sms > 0: the persistent grid spreads over at most that many SMs
  const int64_t resident =
      static_cast<int64_t>(max_sms > 0 && max_sms < sms ? max_sms : sms) * ctas_per_sm;
  int64_t runs;
  plan->tile_bound = 0;
  if (partition_tokens > 0) {
    // Runs of at most partition_tokens tokens, as many as every streaming warp of the grid
    // can take in equal numbers (a multiple of the warp count once there are more runs than
    // warps), split evenly over the real tile count: no warp ends a whole run after the rest.
    const int64_t max_tiles = partition_tokens / kBlockSize;
    const int64_t least = (tiles_upper + max_tiles - 1) / max_tiles;
    auto even = [least](int64_t warps) {
      return least > warps ? (least + warps - 1) / warps * warps : least;
    };
    runs = even(resident * kWarps);
    // Under an SM budget, never more runs (partials) than on the whole device, so the
    // workspace the size query returns (which knows no budget) always suffices; the warps
    // then take one run more or less each.
    const int64_t runs_full = even(static_cast<int64_t>(sms) * ctas_per_sm * kWarps);
    if (runs > runs_full) runs = runs_full;
    plan->chunk = 0;
    plan->tile_bound = tiles_upper;
  } else {
    plan->chunk = 0;
    runs = resident * kWarps;
    const int64_t by_size = (tiles_upper + kMinTilesPerRun - 1) / kMinTilesPerRun;
    if (by_size < runs) runs = by_size;
    // One short sequence: one CTA per K/V head.  Its tiles (num_kv_heads segments of equal
    // length) split into num_kv_heads * kWarps equal runs put every segment's pieces on
    // one CTA, so they publish and merge with CTA-scope ordering instead of device-scope
    // fences.
    if (num_seqs == 1 && num_kv_heads <= resident &&
        tiles_upper <= static_cast<int64_t>(kOneSeqMaxTilesPerWarp) * num_kv_heads * kWarps)
      runs = static_cast<int64_t>(num_kv_heads) * kWarps;
  }
  if (runs < 1) runs = 1;
  if (runs > 0x7fffffff) return cudaErrorInvalidValue;
  plan->runs = static_cast<int>(runs);
  const int64_t ctas = (runs + kWarps - 1) / kWarps;
  plan->grid = static_cast<int>(ctas < resident ? ctas : resident);
  plan->fused_merge = partition_tokens == 0 && max_context_len <= kFusedMergeMaxContext;
  // Pieces per (sequence, kv head) segment at the longest context: with many, the merge
  // kernel spreads each segment's query heads over separate CTAs.
  const int64_t seg_pieces =
      partition_tokens > 0 ? (max_context_len + partition_tokens - 1) / partition_tokens
                           : runs / (static_cast<int64_t>(num_seqs) * num_kv_heads) + 2;
  plan->merge_split_heads = !plan->fused_merge && seg_pieces >= kMergeSplitPieces;
  // Under an SM budget another kernel shares DRAM and L2 with this one: no extra requests.
  plan->prefetch_ok = !(max_sms > 0 && max_sms < sms);
  plan->ws_count_offset = (16 + sizeof(int32_t) * (num_seqs + 1) + 255) / 256 * 256;
  plan->ws_meta_bytes = plan->ws_count_offset +
                        (sizeof(int32_t) * num_seqs * num_kv_heads + 255) / 256 * 256;
  plan->workspace_bytes = plan->ws_meta_bytes +
                          static_cast<size_t>(runs) * 2 * group * kPartialFloats * sizeof(float);
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
  switch (plan.group) {
    case 1: return launch<1>(a, plan, stream);
    case 2: return launch<2>(a, plan, stream);
    case 4: return launch<4>(a, plan, stream);
    default: return cudaErrorInvalidValue;
  }
}

int decode_max_seqs() { return kMaxSeqs; }

}  // namespace pkv
