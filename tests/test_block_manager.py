"""Host-side block manager (pa_bm_*): on-demand block growth, shared blocks with reference
counts, copy-on-write of a shared partly filled last block, freeing.  Pure host code, so
these tests run without a GPU.  A small Python model of the same rules ("vLLM",
PagedAttention) checks random operation sequences."""
import random

import pytest

from paged_kv_cache_299_gb300 import binding as pa
from _util import read_golden


def test_300_tokens_take_19_blocks_one_at_a_time():
    g = {r[0]: int(r[1]) for r in read_golden("block_arithmetic.txt")}
    bm = pa.BlockManager(64, 16)
    bm.add_sequence(0)
    for t in range(1, g["tokens"] + 1):  # tokens arrive one by one
        assert bm.append_tokens(0, 1) == []
        _, n = bm.block_table(0, 64)
        assert n == -(-t // 16)  # a new block exactly when the previous one is full
    _, n = bm.block_table(0, 64)
    assert n == g["blocks"] and bm.num_free_blocks == 64 - g["blocks"]
    assert g["blocks"] * 16 - bm.num_tokens(0) == g["wasted_slots"]


def test_fork_shares_blocks_and_copies_on_first_write_only():
    bm = pa.BlockManager(16, 16)
    bm.add_sequence(1)
    bm.append_tokens(1, 40)  # 3 blocks, last one has 8 tokens
    table, n = bm.block_table(1, 8)
    bm.fork(1, 2)
    assert bm.block_table(2, 8) == (table, n)
    assert all(bm.ref_count(b) == 2 for b in table[:n])
    free = bm.num_free_blocks
    pairs = bm.append_tokens(1, 1)  # writes into the shared last block -> copy it
    assert len(pairs) == 1 and pairs[0][0] == table[n - 1]
    t1, _ = bm.block_table(1, 8)
    assert t1[:n - 1] == table[:n - 1] and t1[n - 1] == pairs[0][1]
    assert bm.ref_count(table[n - 1]) == 1 and bm.num_free_blocks == free - 1
    assert bm.append_tokens(2, 1) == []  # the other sharer now owns the block alone
    assert bm.block_table(2, 8)[0] == table
    bm.free_sequence(1)
    bm.free_sequence(2)
    assert bm.num_free_blocks == 16


def test_full_shared_block_needs_no_copy():
    bm = pa.BlockManager(8, 16)
    bm.add_sequence(0)
    bm.append_tokens(0, 32)
    bm.fork(0, 1)
    assert bm.append_tokens(0, 5) == [] and bm.append_tokens(1, 5) == []
    t0, n0 = bm.block_table(0, 8)
    t1, n1 = bm.block_table(1, 8)
    assert n0 == n1 == 3 and t0[:2] == t1[:2] and t0[2] != t1[2]


def test_out_of_blocks_changes_nothing():
    bm = pa.BlockManager(3, 16)
    bm.add_sequence(0)
    bm.append_tokens(0, 20)
    before = (bm.block_table(0, 4), bm.num_free_blocks, bm.num_tokens(0))
    with pytest.raises(pa.PagedKVError) as e:
        bm.append_tokens(0, 40)  # needs 3 more blocks, 1 free
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    assert (bm.block_table(0, 4), bm.num_free_blocks, bm.num_tokens(0)) == before


def test_bad_calls_are_rejected():
    bm = pa.BlockManager(4, 16)
    bm.add_sequence(0)
    for call in (lambda: bm.add_sequence(0), lambda: bm.fork(7, 1), lambda: bm.fork(0, 0),
                 lambda: bm.free_sequence(5), lambda: bm.append_tokens(9, 1)):
        with pytest.raises(pa.PagedKVError):
            call()
    assert bm.num_tokens(42) == -1 and bm.ref_count(99) == -1


class Model:
    def __init__(self, nb, bs):
        self.bs, self.free, self.ref, self.seqs = bs, list(range(nb - 1, -1, -1)), [0] * nb, {}

    def add(self, s):
        self.seqs[s] = ([], 0)

    def fork(self, p, c):
        blocks, t = self.seqs[p]
        for b in blocks:
            self.ref[b] += 1
        self.seqs[c] = (list(blocks), t)

    def append(self, s, n):
        blocks, t = self.seqs[s]
        need = -(-(t + n) // self.bs)
        cow = t % self.bs != 0 and blocks and self.ref[blocks[-1]] > 1
        if (need - len(blocks)) + (1 if cow else 0) > len(self.free):
            return None
        pairs = []
        if cow:
            b = self.free.pop()
            self.ref[b] = 1
            self.ref[blocks[-1]] -= 1
            pairs.append((blocks[-1], b))
            blocks[-1] = b
        while len(blocks) < need:
            b = self.free.pop()
            self.ref[b] = 1
            blocks.append(b)
        self.seqs[s] = (blocks, t + n)
        return pairs

    def drop(self, s):
        for b in self.seqs.pop(s)[0]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)


@pytest.mark.parametrize("seed", range(5))
def test_random_operations_match_the_model(seed):
    rng = random.Random(seed)
    nb = 40
    bm, model = pa.BlockManager(nb, 16), Model(nb, 16)
    next_id = 0
    for _ in range(400):
        op = rng.random()
        live = list(model.seqs)
        if op < 0.15 or not live:
            bm.add_sequence(next_id)
            model.add(next_id)
            next_id += 1
        elif op < 0.3:
            p = rng.choice(live)
            bm.fork(p, next_id)
            model.fork(p, next_id)
            next_id += 1
        elif op < 0.8:
            s = rng.choice(live)
            n = rng.choice([1, 1, 2, 7, 16, 30])
            want = model.append(s, n)
            if want is None:
                with pytest.raises(pa.PagedKVError):
                    bm.append_tokens(s, n)
            else:
                assert bm.append_tokens(s, n) == want
        else:
            s = rng.choice(live)
            bm.free_sequence(s)
            model.drop(s)
        assert bm.num_free_blocks == len(model.free)
        for s, (blocks, t) in model.seqs.items():
            table, n = bm.block_table(s, nb)
            assert table[:n] == blocks and bm.num_tokens(s) == t
        assert all(bm.ref_count(b) == model.ref[b] for b in range(nb))
