"""Pins of the CPU oracle against facts fixed by the pages or by mathematics.

Each test names the mistake it would catch.  The oracle is compared with: the pages'
block arithmetic and GQA figure (golden files), a hand-worked block-table example,
numpy indexing of the pool layout, torch's scaled_dot_product_attention in float64
(a library routine, not the oracle's formula retyped), closed forms and invariants.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_299_gb300 import workloads as wl
from _util import dense_kv, oracle_pools, read_golden, sdpa_decode


# ---- block arithmetic and slot mapping ------------------------------------------------

def test_block_arithmetic_golden():
    g = {r[0]: int(r[1]) for r in read_golden("block_arithmetic.txt")}
    assert oracle.blocks_for_tokens(g["tokens"], g["block_size"]) == g["blocks"]
    assert oracle.blocks_for_tokens(g["blocks"] * 16, 16) == g["blocks"]
    assert oracle.blocks_for_tokens(1, 16) == 1 and oracle.blocks_for_tokens(0, 16) == 0


def test_300_tokens_fill_19_blocks_and_leave_4_slots():
    """Store a 300-token sequence through the oracle: exactly 19 physical blocks are
    touched and exactly 4 slots (per head) of the last one keep their sentinel."""
    g = {r[0]: int(r[1]) for r in read_golden("block_arithmetic.txt")}
    w = wl.single_sequence_300()
    vals = w.values(0, "cpu")
    kc, vc = oracle_pools(w, vals)
    touched = ~np.all(kc == wl.NAN_BF16, axis=(1, 2, 3))
    assert touched.sum() == g["blocks"]
    assert set(np.nonzero(touched)[0]) == set(w.block_tables[0, :g["blocks"]].tolist())
    last = w.block_tables[0, g["blocks"] - 1]
    per_head_nan_rows = np.all(kc[last] == wl.NAN_BF16, axis=2).sum(axis=1)
    assert np.all(per_head_nan_rows == g["wasted_slots"])


def test_block_table_worked_example():
    rows = {r[0]: [int(x) for x in r[1:]] for r in read_golden("block_table_example.txt")}
    table = np.array([rows["table"]], dtype=np.int32)
    ctx = np.array(rows["context"], dtype=np.int32)
    qsl = np.array([0, ctx[0]], dtype=np.int32)
    slots, err = oracle.slot_mapping(table, ctx, qsl, num_blocks=8)
    assert err == 0
    assert slots.tolist() == rows["slots"]
    # Appending one token to a 35-token context (decode) lands at position 34.
    slots, err = oracle.slot_mapping(table, ctx, np.array([0, 1], np.int32), num_blocks=8)
    assert err == 0 and slots.tolist() == [rows["slots"][-1]]


def test_slot_mapping_rejects_bad_entries():
    table = np.array([[3, -1]], dtype=np.int32)
    slots, err = oracle.slot_mapping(table, np.array([20], np.int32),
                                     np.array([0, 20], np.int32), num_blocks=4)
    assert err == oracle.BAD_BLOCK and (slots[16:] == -1).all() and (slots[:16] >= 48).all()
    slots, err = oracle.slot_mapping(table, np.array([40], np.int32),
                                     np.array([0, 1], np.int32), num_blocks=4)
    assert err == oracle.BAD_POSITION and slots[0] == -1


# ---- scatter --------------------------------------------------------------------------

def test_scatter_layout_matches_numpy_indexing():
    """Token t lands in pool[slot // 16, :, slot % 16, :] (the [NB, Hkv, 16, D] layout,
    read back with numpy indexing); everything else keeps its sentinel."""
    rng = np.random.default_rng(7)
    nb, t = 10, 37
    slots = rng.permutation(nb * 16)[:t].astype(np.int64)
    slots[5] = -1  # skipped
    k = rng.integers(0, 2**16, size=(t, 8, 64), dtype=np.uint16)
    v = rng.integers(0, 2**16, size=(t, 8, 64), dtype=np.uint16)
    kc, vc = wl.nan_pool(nb), wl.nan_pool(nb)
    assert oracle.reshape_and_cache(k, v, slots, kc, vc) == 0
    written = np.zeros((nb, 16), dtype=bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(kc[s // 16, :, s % 16, :], k[i])
        assert np.array_equal(vc[s // 16, :, s % 16, :], v[i])
        written[s // 16, s % 16] = True
    assert np.all(kc.transpose(0, 2, 1, 3)[~written] == wl.NAN_BF16)
    assert np.all(vc.transpose(0, 2, 1, 3)[~written] == wl.NAN_BF16)


# ---- attention against a library routine ----------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_decode_matches_sdpa(seed):
    """Catches a dropped scale, a sign error, a transposed operand, a wrong GQA index and
    any paging mistake: the reference sees contiguous K/V, the oracle the paged pool."""
    w = wl.random_small(seed, num_seqs=4, max_ctx=70)
    vals = w.values(0, "cpu")
    kc, vc = oracle_pools(w, vals)
    out, err = oracle.decode(wl.bf16_bits(vals["q_decode"]), kc, vc, w.block_tables,
                             w.context_lens, w.scale)
    assert err == 0
    for s in range(w.num_decode):
        ref = sdpa_decode(w, vals, s).numpy()
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [10, 11, 12])
def test_prefill_matches_sdpa_causal_square(seed):
    """Chunk rows equal the last q_len rows of a square causal attention over all L
    positions (torch is_causal on an L x L problem, where its mask is unambiguous).
    Catches causal off-by-one errors and a wrong chunk-position offset."""
    w = wl.random_small(seed, num_seqs=3, max_ctx=60, num_prefill=3, max_chunk=30)
    vals = w.values(0, "cpu")
    kc, vc = oracle_pools(w, vals)
    out, err = oracle.prefill_chunk(wl.bf16_bits(vals["q_prefill"]), w.prefill_query_start_loc,
                                    kc, vc, w.block_tables, w.context_lens, w.scale)
    assert err == 0
    qsl = w.prefill_query_start_loc
    gen = torch.Generator().manual_seed(seed)
    for s in range(w.num_prefill):
        k, v = dense_kv(w, vals, s)
        L = k.shape[1]
        q_len = qsl[s + 1] - qsl[s]
        q_full = torch.randn(32, L, 64, generator=gen, dtype=torch.float64)
        q_full[:, L - q_len:, :] = vals["q_prefill"][qsl[s]:qsl[s + 1]].to(
            torch.float64).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q_full[None], k[None], v[None], is_causal=True, scale=w.scale, enable_gqa=True)
        ref = ref[0, :, L - q_len:, :].transpose(0, 1).numpy()
        np.testing.assert_allclose(out[qsl[s]:qsl[s + 1]], ref, rtol=0, atol=1e-12)


def test_group_of_one_is_plain_multi_head_attention():
    """With as many K/V heads as query heads the method is standard MHA."""
    rng = np.random.default_rng(3)
    L, H, D = 23, 8, 64
    k = torch.randn(H, L, D, dtype=torch.float64).to(torch.bfloat16)
    v = torch.randn(H, L, D, dtype=torch.float64).to(torch.bfloat16)
    q = torch.randn(1, H, D, dtype=torch.float64).to(torch.bfloat16)
    table = rng.permutation(4).astype(np.int32)[None, :2]
    kc = np.full((4, H, 16, D), wl.NAN_BF16, np.uint16)
    vc = kc.copy()
    slots, err = oracle.slot_mapping(table, np.array([L], np.int32),
                                     np.array([0, L], np.int32), 4)
    assert err == 0
    assert oracle.reshape_and_cache(wl.bf16_bits(k.transpose(0, 1)),
                                    wl.bf16_bits(v.transpose(0, 1)), slots, kc, vc) == 0
    out, err = oracle.decode(wl.bf16_bits(q), kc, vc, table, np.array([L], np.int32), 0.125)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.to(torch.float64)[:, :, None, :], k.to(torch.float64)[None],
        v.to(torch.float64)[None], scale=0.125)[0, :, 0, :]
    np.testing.assert_allclose(out[0], ref.numpy(), rtol=0, atol=1e-12)


# ---- closed forms and special cases ---------------------------------------------------

def _single_seq(L, seed=0, kv=None):
    w = wl.make_workload("t", [0], [L], seed=seed, pool_slack=1.0)
    vals = w.values(0, "cpu")
    if kv is not None:
        vals.update(kv(vals))
    return w, vals


def test_context_of_one_returns_v_exactly():
    w, vals = _single_seq(1)
    kc, vc = oracle_pools(w, vals)
    out, err = oracle.decode(wl.bf16_bits(vals["q_decode"]), kc, vc, w.block_tables,
                             w.context_lens, w.scale)
    v0 = vals["new_v"][0].to(torch.float64).numpy()  # [Hkv, D]
    for h in range(32):
        assert np.array_equal(out[0, h], v0[h // 4])


def test_identical_keys_give_mean_of_values():
    def same_keys(vals):
        k = vals["new_k"].clone()
        k[:] = k[0]
        return {"new_k": k}
    w, vals = _single_seq(45, kv=same_keys)
    kc, vc = oracle_pools(w, vals)
    out, _ = oracle.decode(wl.bf16_bits(vals["q_decode"]), kc, vc, w.block_tables,
                           w.context_lens, w.scale)
    mean_v = vals["new_v"].to(torch.float64).mean(0).numpy()
    for h in range(32):
        np.testing.assert_allclose(out[0, h], mean_v[h // 4], rtol=0, atol=1e-13)


def test_two_keys_logistic_closed_form():
    """softmax over two scores is the logistic function of their difference."""
    w, vals = _single_seq(2, seed=5)
    kc, vc = oracle_pools(w, vals)
    out, _ = oracle.decode(wl.bf16_bits(vals["q_decode"]), kc, vc, w.block_tables,
                           w.context_lens, w.scale)
    k = vals["new_k"].to(torch.float64).numpy()
    v = vals["new_v"].to(torch.float64).numpy()
    q = vals["q_decode"][0].to(torch.float64).numpy()
    for h in range(32):
        g = h // 4
        delta = w.scale * (q[h] @ k[0, g] - q[h] @ k[1, g])
        a = 1.0 / (1.0 + np.exp(-delta))
        np.testing.assert_allclose(out[0, h], a * v[0, g] + (1 - a) * v[1, g], rtol=0,
                                   atol=1e-13)


def test_gqa_mapping_golden():
    """Heads joined to the same K/V head in the figure, given the same query, give the
    same output; heads in different groups do not."""
    pairs = [(int(a), int(b)) for a, b in read_golden("gqa_mapping.txt")[:6]]
    w, vals = _single_seq(33, seed=9)
    q = vals["q_decode"].clone()
    q[0, :] = q[0, 0]  # every head asks the same question
    kc, vc = oracle_pools(w, vals)
    out, _ = oracle.decode(wl.bf16_bits(q), kc, vc, w.block_tables, w.context_lens, w.scale)
    for h, g in pairs:
        for h2, g2 in pairs:
            same = np.array_equal(out[0, h], out[0, h2])
            assert same == (g == g2), (h, h2)


def test_large_scores_stay_finite_and_exact():
    """Keys scaled x8 (scores of tens) must not overflow the softmax."""
    w = wl.make_workload("big", [50, 90], [1, 1], seed=4, pool_slack=0.3,
                         big_key_fraction=0.2)
    vals = w.values(0, "cpu")
    kc, vc = oracle_pools(w, vals)
    out, err = oracle.decode(wl.bf16_bits(vals["q_decode"]), kc, vc, w.block_tables,
                             w.context_lens, w.scale)
    assert err == 0 and np.isfinite(out).all()
    for s in range(2):
        np.testing.assert_allclose(out[s], sdpa_decode(w, vals, s).numpy(), rtol=0, atol=1e-12)


# ---- invariants -----------------------------------------------------------------------

def test_physical_block_permutation_leaves_output_bit_identical():
    w = wl.random_small(21, num_seqs=3, max_ctx=80)
    vals = w.values(0, "cpu")
    kc, vc = oracle_pools(w, vals)
    out, _ = oracle.decode(wl.bf16_bits(vals["q_decode"]), kc, vc, w.block_tables,
                           w.context_lens, w.scale)
    perm = np.random.default_rng(1).permutation(w.num_blocks)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2, _ = oracle.decode(wl.bf16_bits(vals["q_decode"]), kc2, vc2, bt2, w.context_lens,
                            w.scale)
    assert np.array_equal(out, out2)


def test_future_keys_do_not_change_a_chunk_row():
    w = wl.make_workload("c", [20], [12], num_prefill=1, seed=2, pool_slack=1.0)
    vals = w.values(0, "cpu")
    kc, vc = oracle_pools(w, vals)
    args = (wl.bf16_bits(vals["q_prefill"]), w.prefill_query_start_loc)
    out, _ = oracle.prefill_chunk(*args, kc, vc, w.block_tables, w.context_lens, w.scale)
    # Row i sits at position 20 + i.  Overwrite the key/value of position 25 everywhere.
    blk, off = w.block_tables[0, 25 // 16], 25 % 16
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[blk, :, off, :] = 0x4000
    vc2[blk, :, off, :] = 0x4000
    out2, _ = oracle.prefill_chunk(*args, kc2, vc2, w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(out[:5], out2[:5])  # positions 20..24 cannot see position 25
    assert not np.any(np.all(out[5:] == out2[5:], axis=(1, 2)))  # 25..31 can


def test_chunk_of_one_equals_decode_and_last_row_equals_decode():
    w = wl.make_workload("c", [40], [9], num_prefill=1, seed=6, pool_slack=1.0)
    vals = w.values(0, "cpu")
    kc, vc = oracle_pools(w, vals)
    out, _ = oracle.prefill_chunk(wl.bf16_bits(vals["q_prefill"]), w.prefill_query_start_loc,
                                  kc, vc, w.block_tables, w.context_lens, w.scale)
    dec, _ = oracle.decode(wl.bf16_bits(vals["q_prefill"][-1:]), kc, vc, w.block_tables,
                           w.context_lens, w.scale)
    assert np.array_equal(out[-1], dec[0])
    one, _ = oracle.prefill_chunk(wl.bf16_bits(vals["q_prefill"][-1:]),
                                  np.array([0, 1], np.int32), kc, vc, w.block_tables,
                                  w.context_lens, w.scale)
    assert np.array_equal(one[0], dec[0])


def test_zero_context_gives_zeros_and_bad_block_is_reported():
    kc = wl.nan_pool(2)
    out, err = oracle.decode(np.zeros((1, 32, 64), np.uint16), kc, kc,
                             np.array([[0]], np.int32), np.array([0], np.int32), 0.125)
    assert err == 0 and np.all(out == 0)
    out, err = oracle.decode(np.zeros((1, 32, 64), np.uint16), kc, kc,
                             np.array([[5]], np.int32), np.array([3], np.int32), 0.125)
    assert err == oracle.BAD_BLOCK


# ---- copy-on-write block copy -----------------------------------------------------------

def test_copy_blocks_copies_whole_blocks_in_order():
    """Block dst becomes a byte copy of block src in both pools (numpy indexing), pairs
    applied in order; nothing else changes."""
    rng = np.random.default_rng(5)
    kc = rng.integers(0, 2**16, size=(6, 8, 16, 64), dtype=np.uint16)
    vc = rng.integers(0, 2**16, size=(6, 8, 16, 64), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    pairs = [(1, 4), (4, 5), (0, 2)]  # 4 <- 1, then 5 <- (new) 4, then 2 <- 0
    assert oracle.copy_blocks(kc, vc, pairs) == 0
    for pool, orig in ((kc, k0), (vc, v0)):
        assert np.array_equal(pool[4], orig[1]) and np.array_equal(pool[5], orig[1])
        assert np.array_equal(pool[2], orig[0])
        for b in (0, 1, 3):
            assert np.array_equal(pool[b], orig[b])
    assert oracle.copy_blocks(kc, vc, [(0, 9)]) == oracle.BAD_BLOCK


def test_row_range_split_of_chunks_is_bit_identical_to_one_call():
    """The threaded helpers the full-size GPU tests use: rows [a, b) of a chunk, taken as a
    chunk of b - a rows over the first L - q_len + b keys, give bit for bit the rows of one
    whole-batch oracle call (row i sits at position L - q_len + i either way); decode
    slices likewise."""
    from _util import oracle_decode_rows, oracle_prefill_rows
    w = wl.random_small(31, num_seqs=5, max_ctx=400, num_prefill=3, max_chunk=90)
    vals = w.values(0)
    kc, vc = oracle_pools(w, vals)
    q = wl.bf16_bits(vals["q_prefill"])
    qsl = w.prefill_query_start_loc
    whole, err = oracle.prefill_chunk(q, qsl, kc, vc, w.block_tables[:3], w.context_lens[:3],
                                      w.scale)
    assert err == 0
    split = oracle_prefill_rows(q, qsl, kc, vc, w.block_tables[:3], w.context_lens[:3],
                                w.scale, rows_per_task=7)
    assert np.array_equal(whole, split)
    qd = wl.bf16_bits(vals["q_decode"])
    dec, err = oracle.decode(qd, kc, vc, w.decode_block_tables, w.decode_context_lens, w.scale)
    assert err == 0
    assert np.array_equal(dec, oracle_decode_rows(qd, kc, vc, w.decode_block_tables,
                                                  w.decode_context_lens, w.scale,
                                                  seqs_per_task=1))


def test_oracle_handles_other_kv_head_counts():
    """With 2 K/V heads and 8 query heads the oracle's chunk attention equals torch SDPA
    (float64, causal over each chunk's positions) on dense K/V."""
    w = wl.make_workload("hkv2", [30, 5], [12, 20], num_prefill=2, seed=9, pool_slack=0.5,
                         num_kv_heads=2, num_q_heads=8)
    vals = w.values(0)
    kc, vc = oracle_pools(w, vals)
    assert kc.shape[1] == 2
    out, err = oracle.prefill_chunk(wl.bf16_bits(vals["q_prefill"]), w.prefill_query_start_loc,
                                    kc, vc, w.block_tables, w.context_lens, w.scale)
    assert err == 0
    qsl = w.prefill_query_start_loc
    for s in range(2):
        k, v = dense_kv(w, vals, s)  # [Hkv, L, D]
        L = int(w.context_lens[s])
        q_len = int(qsl[s + 1] - qsl[s])
        q = vals["q_prefill"][qsl[s]:qsl[s + 1]].to(torch.float64).transpose(0, 1)  # [Hq, q, D]
        pos = torch.arange(L - q_len, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None], k[None], v[None], attn_mask=mask, scale=w.scale, enable_gqa=True)[0]
        assert np.abs(out[qsl[s]:qsl[s + 1]] - ref.transpose(0, 1).numpy()).max() < 1e-12
