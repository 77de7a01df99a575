"""GPU parity of the copy-on-write block copy, and an end-to-end parallel-sampling step:
a prompt stored once, three forked samples sharing its blocks, each appending its own token
(each writer but the last copies the shared, partly filled block), decode per sample compared with
the oracle on each sample's logical sequence."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import bits, i32
from _util import ATOL_MAX, ATOL_MEAN, errors

pytestmark = pytest.mark.gpu


def test_copy_blocks_is_bit_exact():
    gen = torch.Generator(device="cuda").manual_seed(3)
    nb = 40
    raw = torch.randint(-2**15, 2**15, (2, nb, 8, 16, 64), generator=gen, device="cuda",
                        dtype=torch.int32).to(torch.int16)
    kc, vc = raw[0].view(torch.bfloat16).contiguous(), raw[1].view(torch.bfloat16).contiguous()
    okc, ovc = bits(kc).copy(), bits(vc).copy()
    perm = np.random.default_rng(4).permutation(nb)
    pairs = np.stack([perm[:12], perm[12:24]], axis=1).astype(np.int64)  # independent pairs
    status = pa.new_device_status()
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda(), device_status=status)
    assert pa.pa_check_device_status(status) == pa.PA_OK
    assert oracle.copy_blocks(okc, ovc, pairs) == 0
    assert np.array_equal(bits(kc), okc) and np.array_equal(bits(vc), ovc)
    bad = torch.tensor([[0, nb + 3]], dtype=torch.int64, device="cuda")
    pa.pa_copy_blocks(kc, vc, bad, device_status=status)
    assert pa.pa_check_device_status(status) == pa.PA_ERR_DEVICE_INDEX
    assert np.array_equal(bits(kc), okc)  # the bad pair was skipped


def test_parallel_sampling_shares_prompt_blocks_with_copy_on_write():
    nb, prompt, samples = 24, 40, 3
    shape = (nb, 8, 16, 64)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(11)
    rnd = lambda *s: torch.randn(*s, generator=gen, device="cuda").to(torch.bfloat16)
    pk, pv = rnd(prompt, 8, 64), rnd(prompt, 8, 64)
    nk, nv = rnd(samples, 8, 64), rnd(samples, 8, 64)
    q = rnd(samples, 32, 64)
    bm = pa.BlockManager(nb, 16)
    maxb = 8
    status = pa.new_device_status()

    def table_of(seqs):
        return i32(np.array([bm.block_table(s, maxb)[0] for s in seqs], np.int32))

    bm.add_sequence(0)
    bm.append_tokens(0, prompt)
    slots = pa.pa_compute_slot_mapping(table_of([0]), i32([prompt]), i32([0, prompt]), prompt,
                                       kc, device_status=status)
    pa.pa_reshape_and_cache(pk, pv, slots, kc, vc, device_status=status)
    for s in range(1, samples):
        bm.fork(0, s)
    used_before = nb - bm.num_free_blocks
    pairs = []
    for s in range(samples):
        pairs += bm.append_tokens(s, 1)
    # every writer but the last holder copies the shared, partly filled last block
    assert len(pairs) == samples - 1 and len({d for _, d in pairs}) == samples - 1
    assert nb - bm.num_free_blocks == used_before + samples - 1
    pa.pa_copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int64, device="cuda"),
                      device_status=status)
    seqs = list(range(samples))
    bt = table_of(seqs)
    ctx = i32([prompt + 1] * samples)
    slots = pa.pa_compute_slot_mapping(bt, ctx, None, samples, kc, device_status=status)
    pa.pa_reshape_and_cache(nk, nv, slots, kc, vc, device_status=status)
    out = torch.empty_like(q)
    pa.pa_decode(out, q, kc, vc, bt, ctx, 0.125, prompt + 1, device_status=status)
    assert pa.pa_check_device_status(status) == pa.PA_OK

    # Oracle: each sample's logical sequence (prompt + its own token) in a private pool.
    for s in range(samples):
        L = prompt + 1
        okc, ovc = wl.nan_pool(4), wl.nan_pool(4)
        table = np.array([[0, 1, 2, 3]], np.int32)
        osl, err = oracle.slot_mapping(table, np.array([L], np.int32), np.array([0, L], np.int32), 4)
        assert err == 0
        k = torch.cat([pk, nk[s:s + 1]])
        v = torch.cat([pv, nv[s:s + 1]])
        oracle.reshape_and_cache(bits(k), bits(v), osl, okc, ovc)
        ref, err = oracle.decode(bits(q[s:s + 1]), okc, ovc, table, np.array([L], np.int32), 0.125)
        assert err == 0
        mx, mean = errors(out[s:s + 1].float().cpu().numpy(), ref)
        assert mx <= ATOL_MAX and mean <= ATOL_MEAN, (s, mx, mean)
