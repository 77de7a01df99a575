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
//   * One CTA per (32-token query tile, K/V head, sequence), two CTAs per SM.  Its 128 MMA
//     rows are the 32 tokens x 4 query heads that share the K/V head (row = 4 * token +
//     head), so each K/V tile feeds four heads.  The query-tile index is the slowest grid
//     dimension, reversed, so the tiles with the longest causal spans start first.
//   * Warp 5 loads the Q tile with one 3-D TMA box and gathers every 64-key K/V tile as
//     four 16-row TMA boxes at the physical blocks named by the block table (128-byte
//     swizzle), into a 4-stage ring; the block table is read in prefetched 32-entry windows.
//   * Warp 4 (one thread) issues S = Q K^T (M128 N64 K64 into one of two fp32 S buffers,
//     so the next tile's scores are computed during this tile's softmax) and
//     [O | l] += P [V | 1] (M128 N80 K64, V read N-major): 16 extra columns of the B operand
//     come from a constant shared-memory atom of bf16 ones, one leading-byte offset from
//     each V slice, so the tensor core also accumulates the row sums l of exactly the bf16
//     P that weights V.  Both A operands come from TMEM: Q is copied there once by the row
//     warps and P is written per tile over the first half of its own S buffer, so each MMA
//     streams only its K or V tile from shared memory.
//   * Warps 0-3 own one TMEM lane = one query row each: they read S, mask by absolute
//     position (diagonal tiles only), keep the running max in registers ([O | l] in TMEM is
//     rescaled only when the max grows by more than 2^8), write P as packed bf16 into TMEM,
//     and finally divide O by l and store bf16 rows.
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
constexpr int kNumBars = 1 + 2 * kStages + 2 + 4; // q, kv full/empty, s x2, p, o, drain, q_tmem
constexpr int kSmemBytes = kQBytes + 2 * kStages * kKVBytes + kOnesBytes + 8 * 16 + 16 + 16;
static_assert(kNumBars <= 16, "barrier area");
static_assert(32 % kBlocksPerTile == 0, "block-table windows hold whole K/V tiles");
// Two CTAs fit on one SM (2 x (kSmemBytes + 1 KiB reserved) <= 228 KiB, 2 x 256 TMEM
// columns = 512, <= 168 registers per thread), so one CTA's softmax overlaps the other's MMAs.
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kSCol = 0;     // two S buffers (fp32): columns 0..63 and 64..127; P (bf16
                                  // pairs) of a tile overwrites the first 32 of its S buffer
constexpr uint32_t kOCol = 128;   // O (fp32): columns 128..191, then 16 row-sum columns
constexpr uint32_t kLCol = kOCol + kHeadDim;  // row sum l (columns 192..207 hold 16 copies)
constexpr uint32_t kQCol = 224;   // Q (bf16 pairs): columns 224..255, the A operand of S = Q K^T
constexpr int kPVN = kHeadDim + 16;  // PV MMA width: 64 output dims + 16 ones columns
constexpr int kThreads = 192;
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
  // Work-list mode (unified varlen launch): CTA b serves item b / num_kv_heads, KV head
  // b % num_kv_heads; items are (sequence, query tile) pairs, heaviest first.
  const int32_t* items;
  const int32_t* item_count;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* status) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  flag_error(status, PA_DEVFLAG_TIMEOUT);
  *abort_flag = 1;
  return false;
}

__global__ void __launch_bounds__(kThreads, 2)
paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const PParams p) {
  int tile, g, s;
  if (p.items != nullptr) {
    const int item = static_cast<int>(blockIdx.x) / p.num_kv_heads;
    if (item >= *p.item_count) return;
    s = p.items[2 * item];
    tile = p.items[2 * item + 1];
    g = static_cast<int>(blockIdx.x) % p.num_kv_heads;
  } else {
    // The query-tile index is the slowest grid dimension, reversed: the tiles with the
    // longest causal spans of every sequence and head are dispatched first.
    tile = gridDim.z - 1 - blockIdx.z;
    g = blockIdx.y;
    s = blockIdx.x;
  }
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int q0 = p.query_start_loc[s];
  const int q_len = p.query_start_loc[s + 1] - q0;
  const int tok0 = tile * kTokensPerTile;
  if (tok0 >= q_len) return;
  if (q0 < 0 || q0 + q_len > p.num_query_tokens) {  // rows outside q / out
    if (tid == 0) flag_error(p.status, PA_DEVFLAG_BAD_CONTEXT);
    return;
  }
  const int L = p.context_lens[s];
  if (L < q_len || static_cast<int64_t>(L) > static_cast<int64_t>(p.max_blocks_per_seq) * kBlockSize) {
    if (tid == 0) flag_error(p.status, PA_DEVFLAG_BAD_CONTEXT);
    return;
  }
  const int ntok = min(kTokensPerTile, q_len - tok0);
  // Row warp w holds tokens tok0 + 8w .. +7; a warp with none of them inside the chunk
  // (every warp but the first for a decode row) skips the softmax entirely: the rows it
  // would produce are discarded, and MMA rows are independent.
  const int live_warps = min(4, (ntok + kTokensPerTile / 4 - 1) / (kTokensPerTile / 4));
  const int keys = L - q_len + tok0 + ntok;  // this tile needs keys 0 .. keys-1
  const int n_kv = (keys + kTileN - 1) / kTileN;
  const int blocks_needed = (keys + kBlockSize - 1) / kBlockSize;

  extern __shared__ __align__(1024) uint8_t smem[];  // 128-byte swizzle atoms need 1 KiB
  if ((smem_addr(smem) & 1023u) != 0) {  // never issue swizzled copies to a misaligned tile
    if (tid == 0) flag_error(p.status, PA_DEVFLAG_LAYOUT);
    return;
  }
  uint8_t* sq = smem;
  uint8_t* sk = sq + kQBytes;
  uint8_t* sv = sk + kStages * kKVBytes;
  uint8_t* sones = sv + kStages * kKVBytes;  // 1 KiB aligned (whole tiles before it)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sones + kOnesBytes);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_ready = kv_empty + kStages;  // [2]
  uint64_t* p_ready = s_ready + 2;
  uint64_t* o_done = p_ready + 1;
  uint64_t* drain = o_done + 1;
  uint64_t* q_tmem = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int& abort_flag = *reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(&s_ready[0], 1);
    mbar_init(&s_ready[1], 1);
    mbar_init(p_ready, 32 * live_warps);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(q_tmem, 32 * live_warps);
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
  // The ones atom: every bf16 of it is 1.0, so the 16 extra columns of O += P [V | 1] each
  // accumulate the row sum of P, exactly the bf16 values that weight V.
  for (int i = tid; i < kOnesBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(sones)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async_smem();  // generic writes before the tensor core's reads
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 5) {
    // ================================ TMA producer ================================
    const int32_t* row = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, kQBytes);
      tma_load_3d(sq, &tmap_q, 0, g * kGroup, q0 + tok0, q_full);
    }
    // The block table is read 32 entries (eight K/V tiles) at a time, one entry per lane,
    // with the next window already in flight, so no tile waits on a block-table load.
    auto fetch = [&](int base) -> int32_t {
      return base + lane < blocks_needed ? __ldg(row + base + lane) : 0;
    };
    int win_base = 0;
    int32_t win = fetch(0);
    int32_t win_next = fetch(32);
    int issued = 0;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j % kStages;
      const int lb0 = j * kBlocksPerTile;
      if (lb0 >= win_base + 32) {
        win_base += 32;
        win = win_next;
        win_next = fetch(win_base + 32);
      }
      const int lb = lb0 + lane;
      const bool need = lane < kBlocksPerTile && lb < blocks_needed;
      const int32_t entry =
          __shfl_sync(0xffffffffu, win, (lb0 - win_base) + (lane & (kBlocksPerTile - 1)));
      const int32_t phys = need ? entry : 0;
      const bool bad = need && (phys < 0 || phys >= p.num_blocks);
      const bool load = need && !bad;
      const unsigned mask = __ballot_sync(0xffffffffu, load);
      const unsigned bad_mask = __ballot_sync(0xffffffffu, bad);
      if (lane == 0 && bad_mask != 0) flag_error(p.status, PA_DEVFLAG_BAD_BLOCK);
      int ok = 1;
      if (lane == 0) {
        ok = wait_or_abort(&kv_empty[st], static_cast<uint32_t>((j / kStages) & 1) ^ 1u,
                           &abort_flag, p.status);
        if (ok) mbar_arrive_expect_tx(&kv_full[st], __popc(mask) * 2u * kTileBytes);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (load) {
        const int y = (phys * p.num_kv_heads + g) * kBlockSize;
        tma_load_2d(sk + st * kKVBytes + lane * kTileBytes, &tmap_k, 0, y, &kv_full[st]);
        tma_load_2d(sv + st * kKVBytes + lane * kTileBytes, &tmap_v, 0, y, &kv_full[st]);
      }
      ++issued;
    }
    // leave no copy in flight: wait (bounded) for the Q tile and the last fill per stage
    if (lane == 0) {
      if (!mbar_wait(q_full, 0)) flag_error(p.status, PA_DEVFLAG_TIMEOUT);
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / kStages) * kStages;
        if (!mbar_wait(&kv_full[st], static_cast<uint32_t>((last / kStages) & 1)))
          flag_error(p.status, PA_DEVFLAG_TIMEOUT);
      }
    }
  } else if (warp == 4) {
    // ================================ MMA issuer ==================================
    // Both A operands live in tensor memory (Q copied there once, P written there by the
    // row warps over its tile's scores), so each MMA streams only its B tile (K or V,
    // 2 KiB per K16 step) from shared memory.  Order: S(0), S(1), PV(0), S(2), PV(1), ...:
    // the scores of the next tile are on the tensor core while the row warps run the
    // softmax of the current one; S(j+2) reuses the buffer of P(j) only after PV(j) (the
    // tensor core runs one thread's MMAs in order).
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTileM, kTileN, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kTileM, kPVN, true);
      const uint32_t ones_addr = smem_addr(sones);
      auto issue_s = [&](int j) -> bool {
        const int st = j % kStages;
        if (!wait_or_abort(&kv_full[st], static_cast<uint32_t>((j / kStages) & 1), &abort_flag,
                           p.status))
          return false;
        tc_fence_after_sync();
        const uint32_t k_base = smem_addr(sk + st * kKVBytes);
        const uint32_t s_tmem = tmem + kSCol + (j & 1) * kTileN;
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          umma_bf16_ts(s_tmem, tmem + kQCol + kk * 8, sw128_desc(k_base + kk * 32, 16, 1024),
                       kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_ready[j & 1]);
        return true;
      };
      auto issue_pv = [&](int j) {
        const uint32_t v_base = smem_addr(sv + (j % kStages) * kKVBytes);
        const uint32_t p_tmem = tmem + kSCol + (j & 1) * kTileN;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          // B = [V rows kk*16 .. +15 | ones]: output dims 0..63 from the V tile (N-major,
          // 128-byte swizzle), columns 64..79 from the ones atom, one leading-byte offset away
          const uint32_t b_addr = v_base + kk * 16 * kRowBytes;
          const uint64_t b = sw128_desc(b_addr, ones_addr - b_addr, 1024);
          umma_bf16_ts(tmem + kOCol, p_tmem + kk * 8, b, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(o_done);
        umma_commit(&kv_empty[j % kStages]);
      };
      bool ok = wait_or_abort(q_tmem, 0, &abort_flag, p.status);
      if (ok) {
        tc_fence_after_sync();
        ok = issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv && !issue_s(j + 1)) break;  // S buffer (j+1)&1 was freed by P(j-1)
        if (!wait_or_abort(p_ready, static_cast<uint32_t>(j & 1), &abort_flag, p.status)) break;
        tc_fence_after_sync();
        issue_pv(j);
      }
      // wait (bounded) until every MMA issued above has completed
      umma_commit(drain);
      if (!mbar_wait(drain, 0)) flag_error(p.status, PA_DEVFLAG_TIMEOUT);
    }
  } else if (warp < live_warps) {
    // ============================ softmax / epilogue (warps 0-3) ============================
    const int r = tid;  // MMA row == TMEM lane
    const int tt = r >> 2;
    const int hh = r & 3;
    const int token = tok0 + tt;
    const bool row_ok = token < q_len;
    const int pos = L - q_len + min(token, q_len - 1);
    const int pos_lo = L - q_len + tok0;  // smallest position among this CTA's rows
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m = -INFINITY;
    bool ok = wait_or_abort(q_full, 0, &abort_flag, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      // copy this row of the (128-byte swizzled) Q tile into tensor memory
      uint32_t qv[32];
      const uint8_t* qrow = sq + r * kRowBytes;
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
      mbar_arrive(q_tmem);
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      ok = wait_or_abort(&s_ready[j & 1], static_cast<uint32_t>((j >> 1) & 1), &abort_flag,
                         p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const int kb = j * kTileN;
      const uint32_t s_addr = lane_addr + kSCol + (j & 1) * kTileN;
      uint32_t v[2][32];  // raw scores; then, in place in v[0], packed bf16 probabilities
      tmem_ld32(s_addr, v[0]);
      tmem_ld32(s_addr + 32, v[1]);
      tmem_wait_ld();
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
      if (j == n_kv - 1 && kb + kTileN > keys) {
        // V rows past the last needed key are never weighted, but may hold NaN (unused
        // slots) or stale data: zero them so 0 * V stays 0 in the tensor core.  The live
        // row warps share the 64 rows.
        for (int zr = r; zr < kTileN; zr += 32 * live_warps) {
          if (kb + zr < keys) continue;
          uint4* vrow = reinterpret_cast<uint4*>(sv + (j % kStages) * kKVBytes + zr * kRowBytes);
#pragma unroll
          for (int i = 0; i < kRowBytes / 16; ++i) vrow[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      if (j > 0) {
        // Every phase of o_done is observed in order (a parity wait cannot tell phases two
        // apart).  PV(j-1) is done with O and its row sum before they are rescaled; P(j)
        // itself needs no wait: PV(j-2), the last reader of this S buffer, completed before
        // S(j) did.
        ok = wait_or_abort(o_done, static_cast<uint32_t>((j - 1) & 1), &abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();
      }
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
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
      tmem_st32(lane_addr + kSCol + (j & 1) * kTileN, v[0]);  // P(j) over S(j)
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(p_ready);
    }
    if (ok) {
      ok = wait_or_abort(o_done, static_cast<uint32_t>((n_kv - 1) & 1), &abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after_sync();
      __syncwarp();
      const uint32_t lsum = tmem_ld1(lane_addr + kLCol);
      tmem_wait_ld();
      const float inv = 1.f / __uint_as_float(lsum);  // l >= 1: the max key weighs >= 1
      __nv_bfloat16* dst = p.out + (static_cast<int64_t>(q0 + token) * p.num_q_heads +
                                    g * kGroup + hh) * kHeadDim;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // 32 columns at a time keeps the register budget
        uint32_t o[32];
        tmem_ld32(lane_addr + kOCol + 32 * c, o);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = q4 * 8 + 2 * e;
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[i]) * inv,
                                                              __uint_as_float(o[i + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * q4) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
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

// [rows][64] bf16 tensor read in boxes of `box_rows` rows (128-byte swizzle).
bool encode_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
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
      !encode_rows(tk, a.key_cache, pool_rows, kBlockSize) ||
      !encode_rows(tv, a.value_cache, pool_rows, kBlockSize))
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
  p->items = nullptr;
  p->item_count = nullptr;
  return cudaSuccess;
}

// ---- work list of the unified varlen launch ---------------------------------------------
// Items are (sequence, 32-token query tile) pairs; an item's work is its number of 64-key
// tiles.  One CTA counting-sorts them by work, heaviest first, so the long causal spans
// and long decode contexts start before the short ones and the launch ends without a long
// tail.  Items of one work value keep no particular order (outputs do not depend on it).
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 4096;  // work values >= 4095 tiles share the last bucket

__device__ __forceinline__ int plan_bucket(int L, int q_len, int t) {
  const int ntok = min(kTokensPerTile, q_len - t * kTokensPerTile);
  const int keys = max(1, L - q_len + t * kTokensPerTile + ntok);
  return min((keys + kTileN - 1) / kTileN, kPlanBuckets - 1);
}

__global__ void __launch_bounds__(kPlanThreads)
varlen_plan_kernel(const int32_t* query_start_loc, const int32_t* context_lens, int num_seqs,
                   int num_query_tokens, int max_items, int32_t* items, int32_t* item_count,
                   int32_t* status) {
  __shared__ int hist[kPlanBuckets];  // counts, then (after the scan) next free position
  __shared__ int warp_total[kPlanThreads / 32];
  __shared__ int grand_total;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int kWarps = kPlanThreads / 32;
  for (int b = tid; b < kPlanBuckets; b += kPlanThreads) hist[b] = 0;
  __syncthreads();
  // histogram of item work; a sequence's tiles are spread over the lanes of one warp
  for (int s = warp; s < num_seqs; s += kWarps) {
    const int q0 = query_start_loc[s];
    const int q_len = query_start_loc[s + 1] - q0;
    if (q_len == 0) continue;
    if (q_len < 0 || q0 < 0 || q0 + q_len > num_query_tokens) {  // rows outside q / out
      if (lane == 0) flag_error(status, PA_DEVFLAG_BAD_CONTEXT);
      continue;
    }
    const int L = context_lens[s];
    const int tiles = (q_len + kTokensPerTile - 1) / kTokensPerTile;
    for (int t = lane; t < tiles; t += 32) atomicAdd(&hist[plan_bucket(L, q_len, t)], 1);
  }
  __syncthreads();
  // exclusive scan from the heaviest bucket down: thread i owns buckets 4095-4i .. 4092-4i
  constexpr int kPer = kPlanBuckets / kPlanThreads;
  int local[kPer];
  int sum = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    local[k] = hist[kPlanBuckets - 1 - (kPer * tid + k)];
    sum += local[k];
  }
  int incl = sum;  // inclusive scan within the warp
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_total[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_total[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    warp_total[lane] = w;  // inclusive over warps
    if (lane == 31) grand_total = w;
  }
  __syncthreads();
  int start = (warp > 0 ? warp_total[warp - 1] : 0) + incl - sum;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    hist[kPlanBuckets - 1 - (kPer * tid + k)] = start;
    start += local[k];
  }
  __syncthreads();
  for (int s = warp; s < num_seqs; s += kWarps) {
    const int q0 = query_start_loc[s];
    const int q_len = query_start_loc[s + 1] - q0;
    if (q_len <= 0 || q0 < 0 || q0 + q_len > num_query_tokens) continue;
    const int L = context_lens[s];
    const int tiles = (q_len + kTokensPerTile - 1) / kTokensPerTile;
    for (int t = lane; t < tiles; t += 32) {
      const int pos = atomicAdd(&hist[plan_bucket(L, q_len, t)], 1);
      if (pos < max_items) {
        items[2 * pos] = s;
        items[2 * pos + 1] = t;
      }
    }
  }
  if (tid == 0) {
    *item_count = min(grand_total, max_items);
    if (grand_total > max_items) flag_error(status, PA_DEVFLAG_BAD_CONTEXT);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  PParams p;
  cudaError_t e = prepare(a, &tq, &tk, &tv, &p);
  if (e != cudaSuccess) return e;
  const int tiles = (a.max_query_len + kTokensPerTile - 1) / kTokensPerTile;
  if (tiles > 65535 || a.num_kv_heads > 65535) return cudaErrorInvalidValue;
  dim3 grid(a.num_seqs, a.num_kv_heads, tiles);
  paged_prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

int64_t varlen_max_items(int32_t num_seqs, int32_t num_query_tokens) {
  return static_cast<int64_t>(num_query_tokens) / kTokensPerTile + num_seqs + 1;
}

size_t varlen_workspace_size(int32_t num_seqs, int32_t num_query_tokens) {
  return 16 + 8 * static_cast<size_t>(varlen_max_items(num_seqs, num_query_tokens));
}

cudaError_t launch_varlen(const PrefillArgs& a, void* workspace, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  PParams p;
  cudaError_t e = prepare(a, &tq, &tk, &tv, &p);
  if (e != cudaSuccess) return e;
  const int64_t max_items = varlen_max_items(a.num_seqs, a.num_query_tokens);
  const int64_t blocks = max_items * a.num_kv_heads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  int32_t* count = static_cast<int32_t*>(workspace);
  int32_t* items = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + 16);
  varlen_plan_kernel<<<1, kPlanThreads, 0, stream>>>(a.query_start_loc, a.context_lens,
                                                     a.num_seqs, a.num_query_tokens,
                                                     static_cast<int>(max_items), items, count,
                                                     a.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  p.items = items;
  p.item_count = count;
  paged_prefill_kernel<<<static_cast<unsigned>(blocks), kThreads, kSmemBytes, stream>>>(tq, tk,
                                                                                        tv, p);
  return cudaGetLastError();
}

}  // namespace pkv
