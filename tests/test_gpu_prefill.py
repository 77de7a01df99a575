"""GPU parity of the tcgen05 chunked-prefill attention against the oracle, through the
C ABI (bf16 output vs double-precision oracle: max-abs 2e-2, mean-abs 2e-3)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep, host_vals, i32, oracle_step
from _util import ATOL_MAX, ATOL_MEAN, errors, oracle_pools, oracle_prefill_rows

pytestmark = pytest.mark.gpu


def check(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    mx, mean = errors(g, ref)
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN, f"{what}: max {mx:.3g} mean {mean:.3g}"


def run(w):
    step = GpuStep(w)
    out = step.prefill()
    assert step.check_status() == pa.PA_OK
    ref = oracle_step(w, host_vals(step.vals))
    return step, out, ref


@pytest.mark.parametrize("seed", range(6))
def test_random_ragged_chunks(seed):
    rng = np.random.default_rng(seed)
    n = 4
    prior = rng.integers(0, 300, size=n)
    chunk = rng.integers(1, 100, size=n)
    w = wl.make_workload(f"pre{seed}", prior, chunk, num_prefill=n, seed=seed, pool_slack=0.3)
    _, out, ref = run(w)
    check(out, ref["prefill"], w.name)


@pytest.mark.parametrize("prior,chunk", [(0, 1), (0, 32), (0, 33), (0, 128), (0, 129),
                                         (16, 16), (127, 1), (128, 128), (200, 97),
                                         (1000, 64), (5, 300)])
def test_boundary_shapes(prior, chunk):
    w = wl.make_workload(f"b{prior}_{chunk}", [prior], [chunk], num_prefill=1, seed=prior + chunk,
                         pool_slack=0.5)
    _, out, ref = run(w)
    check(out, ref["prefill"], w.name)


def test_large_scores_force_rescale():
    """A fifth of the keys x8: the running max jumps between key tiles, so the O held in
    tensor memory must be rescaled."""
    w = wl.make_workload("big", [400, 260], [160, 70], num_prefill=2, seed=3, pool_slack=0.3,
                         big_key_fraction=0.2)
    _, out, ref = run(w)
    check(out, ref["prefill"], w.name)


def test_empty_chunk_in_batch_and_grid_tail():
    """A sequence with q_len 0 between two others: its CTAs exit, the others are right."""
    w = wl.make_workload("mix", [50, 70, 10], [40, 1, 90], num_prefill=3, seed=4, pool_slack=0.5)
    step = GpuStep(w)
    qsl = w.prefill_query_start_loc.copy()
    # remove the middle sequence's single row from the call: q_len becomes 0
    q = torch.cat([step.vals["q_prefill"][: qsl[1]], step.vals["q_prefill"][qsl[2]:]])
    qsl2 = np.array([0, qsl[1], qsl[1], qsl[1] + (qsl[3] - qsl[2])], np.int32)
    ctx = step.ctx.clone()
    out = torch.empty_like(q)
    pa.pa_prefill_chunk(out, q, i32(qsl2), 90, step.kc, step.vc, step.bt, ctx, w.scale,
                        device_status=step.status)
    assert step.check_status() == pa.PA_OK
    ref = oracle_step(w, host_vals(step.vals))["prefill"]
    ref2 = np.concatenate([ref[: qsl[1]], ref[qsl[2]:]])
    check(out, ref2, "empty chunk")


def test_last_chunk_row_matches_decode_kernel():
    w = wl.make_workload("ld", [333], [45], num_prefill=1, seed=8, pool_slack=0.3)
    step = GpuStep(w)
    out = step.prefill()
    dec = torch.empty_like(out[-1:])
    pa.pa_decode(dec, step.vals["q_prefill"][-1:].contiguous(), step.kc, step.vc, step.bt,
                 step.ctx, w.scale, int(w.context_lens.max()))
    assert (out[-1].float() - dec[0].float()).abs().max().item() <= 1.6e-2


def test_config5_prefill_every_row():
    """Mixed-step workload: 8 chunks of 512 over 0..2048 prior tokens.  Every row of every
    chunk (all 16 query tiles of each), all 32 heads, element by element against the
    oracle's causal chunk attention."""
    w = wl.mixed_prefill_decode()
    step = GpuStep(w)
    out = step.prefill()
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref = oracle_prefill_rows(wl.bf16_bits(hv["q_prefill"]), w.prefill_query_start_loc, kc, vc,
                              w.block_tables[: w.num_prefill], w.context_lens[: w.num_prefill],
                              w.scale)
    assert ref.shape == (4096, 32, 64)
    check(out, ref, "config 5 prefill, every row")


def test_bad_block_is_flagged_not_fatal():
    w = wl.make_workload("bad", [40], [20], num_prefill=1, seed=2, pool_slack=0.5)
    step = GpuStep(w)
    bt = step.bt.clone()
    bt[0, 1] = -7
    status = pa.new_device_status()
    out = torch.empty_like(step.vals["q_prefill"])
    pa.pa_prefill_chunk(out, step.vals["q_prefill"], i32(w.prefill_query_start_loc), 20, step.kc,
                        step.vc, bt, step.ctx, w.scale, device_status=status)
    assert pa.pa_check_device_status(status) == pa.PA_ERR_DEVICE_INDEX
    assert torch.isfinite(step.prefill().float()).all()  # context still usable


def test_long_chunk_every_row():
    """One 4100-row chunk over 4000 prior tokens (129 query tiles, the last one ragged, up
    to 127 key tiles): every row against the oracle's causal chunk attention."""
    w = wl.make_workload("long_chunk", [4000], [4100], num_prefill=1, seed=21, pool_slack=0.1)
    step = GpuStep(w)
    out = step.prefill()
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref = oracle_prefill_rows(wl.bf16_bits(hv["q_prefill"]), w.prefill_query_start_loc, kc, vc,
                              w.block_tables, w.context_lens, w.scale)
    check(out, ref, "long chunk, every row")


def test_many_chunks_beyond_the_in_kernel_sort():
    """2200 short chunks (2..60 rows over 0..120 prior tokens): more (sequence, query tile)
    pairs than the in-kernel sort takes, so the persistent kernel serves its units in grid
    order; every row against the oracle."""
    rng = np.random.default_rng(55)
    n = 2200
    chunk = rng.integers(2, 61, size=n)
    prior = rng.integers(0, 121, size=n)
    w = wl.make_workload("many_chunks", prior, chunk, num_prefill=n, seed=55, pool_slack=0.2)
    pairs = int(((chunk + 31) // 32).sum())
    assert pairs > 2048
    step = GpuStep(w)
    out = step.prefill()
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref = oracle_prefill_rows(wl.bf16_bits(hv["q_prefill"]), w.prefill_query_start_loc, kc, vc,
                              w.block_tables, w.context_lens, w.scale)
    check(out, ref, "many chunks, grid order")


@pytest.mark.parametrize("hkv", [1, 2, 16])
def test_other_kv_head_counts(hkv):
    """Chunks with 1, 2 and 16 K/V heads (4 query heads each): the work units are (query
    tile, K/V head) pairs, so the head count changes how many units each persistent CTA
    serves (16 heads: more units than CTAs).  Every row against the oracle."""
    rng = np.random.default_rng(60 + hkv)
    n = 6
    prior = rng.integers(0, 400, size=n)
    chunk = rng.integers(20, 160, size=n)
    w = wl.make_workload(f"hkv{hkv}", prior, chunk, num_prefill=n, seed=60 + hkv,
                         pool_slack=0.3, num_kv_heads=hkv, num_q_heads=4 * hkv)
    step = GpuStep(w)
    out = step.prefill()
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref = oracle_prefill_rows(wl.bf16_bits(hv["q_prefill"]), w.prefill_query_start_loc, kc, vc,
                              w.block_tables, w.context_lens, w.scale)
    check(out, ref, w.name)
