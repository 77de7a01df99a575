"""GPU parity of the slot mapping, the KV store and paged decode attention against the
oracle, through the C ABI.  Store and slot mapping must be bit-exact; attention must be
within max-abs 2e-2 and mean-abs 2e-3 of the double-precision oracle (bf16 output)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep, bits, host_vals, i32, oracle_step
from _util import ATOL_MAX, ATOL_MEAN, errors

pytestmark = pytest.mark.gpu


def assert_close(got: torch.Tensor, ref: np.ndarray, what=""):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output (a poisoned slot was read)"
    mx, mean = errors(g, ref)
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN, f"{what}: max {mx:.3g} mean {mean:.3g}"


def full_check(w, layer=0, partition_tokens=None):
    step = GpuStep(w, layer)
    out = step.decode(partition_tokens)
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    ref = oracle_step(w, hv)
    # slot mapping and store: bit-exact, sentinels included
    s_ref, err = oracle.slot_mapping(w.block_tables, w.context_lens, w.new_start_loc,
                                     w.num_blocks)
    assert err == 0 and np.array_equal(step.new_slots.cpu().numpy(), s_ref)
    assert np.array_equal(bits(step.kc), ref["kc"]), "key pool differs from the oracle's"
    assert np.array_equal(bits(step.vc), ref["vc"]), "value pool differs from the oracle's"
    assert_close(out, ref["decode"], f"{w.name} decode")
    return step, out, ref


@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("partition_tokens", [0, 16, 64, 512])
def test_small_random_workloads(seed, partition_tokens):
    w = wl.random_small(100 + seed, num_seqs=6, max_ctx=300)
    full_check(w, partition_tokens=partition_tokens)


def test_every_tail_length():
    """Contexts 1..96: every fill of the last block, several blocks."""
    ctx = np.arange(1, 97)
    w = wl.make_workload("tails", ctx - 1, np.ones_like(ctx), seed=5, pool_slack=0.25)
    full_check(w)
    full_check(w, partition_tokens=16)


def test_config1_single_sequence():
    full_check(wl.single_sequence_300())


@pytest.mark.parametrize("L", [1, 17, 300, 768, 769])
def test_single_sequence_one_cta_per_head(L):
    """One sequence of up to 768 tokens (4 tiles per warp) runs one CTA per K/V head, all
    of a head's pieces merged inside its CTA.  At and around that bound, and with a host
    bound of the context above the real one (768: the same plan; 2048: the general one),
    the decode matches the oracle and a reused workspace gives the same bits."""
    w = wl.make_workload(f"one{L}", [L - 1], [1], seed=50 + L, pool_slack=0.5)
    step, _, ref = full_check(w)
    for max_ctx in sorted({L, 768, 2048}):
        if max_ctx < L:
            continue
        ws = torch.zeros(pa.pa_decode_workspace_size(1, 8, 32, max_ctx, 0), dtype=torch.uint8,
                         device="cuda")
        outs = []
        for _ in range(2):
            out = torch.empty_like(step.vals["q_decode"])
            pa.pa_decode(out, step.vals["q_decode"], step.kc, step.vc, step.bt, step.ctx,
                         w.scale, max_ctx, workspace=ws, device_status=step.status)
            outs.append(out)
        assert step.check_status() == pa.PA_OK
        assert torch.equal(outs[0], outs[1])
        assert_close(outs[0], ref["decode"], f"one sequence of {L} tokens, bound {max_ctx}")


def test_config2_decode_batch64():
    full_check(wl.decode_batch64_uniform())


@pytest.mark.parametrize("layer", [0, 15])
def test_config3_decode_batch256_layer(layer):
    full_check(wl.decode_batch256_lognormal(layers=16), layer=layer)


def test_config4_long_context_split512():
    w = wl.long_context_batch4()
    step = GpuStep(w)
    out = step.decode()  # partition_tokens = 512 from the workload
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    ref = oracle_step(w, hv)
    # slot mapping and store of the 4 x 131072 tokens: bit-exact, NaN sentinels included
    s_ref, err = oracle.slot_mapping(w.block_tables, w.context_lens, w.new_start_loc,
                                     w.num_blocks)
    assert err == 0 and np.array_equal(step.new_slots.cpu().numpy(), s_ref)
    assert np.array_equal(bits(step.kc), ref["kc"]), "key pool differs from the oracle's"
    assert np.array_equal(bits(step.vc), ref["vc"]), "value pool differs from the oracle's"
    assert_close(out, ref["decode"], "config 4 decode")
    out_auto = step.decode(0)
    assert_close(out_auto, ref["decode"], "config 4 decode, balanced split")


def test_config5_decode_part():
    w = wl.mixed_prefill_decode()
    step = GpuStep(w)
    out = step.decode()
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = bits(step.kc), bits(step.vc)
    from _util import oracle_pools
    okc, ovc = oracle_pools(w, hv)
    assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)
    ref, err = oracle.decode(wl.bf16_bits(hv["q_decode"]), okc, ovc, w.decode_block_tables,
                             w.decode_context_lens, w.scale)
    assert err == 0
    assert_close(out, ref, "config 5 decode")


def test_split_results_agree():
    """Online softmax over any partition gives the same result (within rounding)."""
    w = wl.random_small(7, num_seqs=5, max_ctx=900)
    step = GpuStep(w)
    outs = [step.decode(p).float() for p in (0, 16, 64, 512, 1024)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1.6e-2


def test_block_permutation_invariance():
    w = wl.random_small(8, num_seqs=4, max_ctx=200)
    step = GpuStep(w)
    out = step.decode()
    perm = torch.from_numpy(np.random.default_rng(3).permutation(w.num_blocks)).cuda()
    kc2 = torch.empty_like(step.kc)
    vc2 = torch.empty_like(step.vc)
    kc2[perm] = step.kc
    vc2[perm] = step.vc
    bt2 = torch.where(step.bt >= 0, perm.to(torch.int32)[step.bt.clamp(min=0).long()], step.bt)
    out2 = torch.empty_like(out)
    pa.pa_decode(out2, step.vals["q_decode"], kc2, vc2, bt2.contiguous(), step.ctx, w.scale,
                 int(w.context_lens.max()))
    assert torch.equal(out, out2)


def test_context_of_one_returns_v_exactly():
    w = wl.make_workload("one", [0, 0, 0], [1, 1, 1], seed=9, pool_slack=1.0)
    step = GpuStep(w)
    out = step.decode()
    v = step.vals["new_v"]  # [3, 8, 64]
    assert torch.equal(out, v.repeat_interleave(4, dim=1))


def test_zero_context_gives_zero_rows():
    w = wl.make_workload("z", [30, 40], [1, 1], seed=2, pool_slack=0.5)
    step = GpuStep(w)
    ctx = step.ctx.clone()
    ctx[1] = 0
    out = torch.full_like(step.vals["q_decode"], 7.0)
    pa.pa_decode(out, step.vals["q_decode"], step.kc, step.vc, step.bt, ctx, w.scale, 41)
    assert torch.count_nonzero(out[1]) == 0
    assert torch.isfinite(out[0].float()).all() and torch.count_nonzero(out[0]) > 0


def test_empty_calls_are_noops():
    kc = torch.zeros(4, 8, 16, 64, dtype=torch.bfloat16, device="cuda")
    empty_kv = torch.empty(0, 8, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_reshape_and_cache(empty_kv, empty_kv, torch.empty(0, dtype=torch.int64, device="cuda"),
                            kc, kc.clone())
    q = torch.empty(0, 32, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_decode(q.clone(), q, kc, kc, torch.empty(0, 1, dtype=torch.int32, device="cuda"),
                 torch.empty(0, dtype=torch.int32, device="cuda"), 0.125, 0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(kc) == 0


def test_negative_slots_are_skipped():
    kc = torch.full((2, 8, 16, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    k = torch.randn(3, 8, 64, device="cuda").to(torch.bfloat16)
    slots = torch.tensor([5, -1, 20], dtype=torch.int64, device="cuda")
    pa.pa_reshape_and_cache(k, k, slots, kc, vc)
    assert torch.equal(kc[0, :, 5], k[0]) and torch.equal(kc[1, :, 4], k[2])
    assert int(torch.isnan(kc.float()).all(dim=-1).sum()) == 2 * 8 * 16 - 2 * 8


def test_device_reports_bad_block_and_bad_context():
    w = wl.make_workload("bad", [20, 20], [1, 1], seed=1, pool_slack=0.5)
    step = GpuStep(w)
    assert step.check_status() == pa.PA_OK
    bt = step.bt.clone()
    bt[1, 0] = w.num_blocks + 5  # out of the pool
    status = pa.new_device_status()
    out = torch.empty_like(step.vals["q_decode"])
    pa.pa_decode(out, step.vals["q_decode"], step.kc, step.vc, bt, step.ctx, w.scale, 21,
                 device_status=status)
    assert pa.pa_check_device_status(status) == pa.PA_ERR_DEVICE_INDEX
    assert int(status.item()) & pa.DEVFLAG_BAD_BLOCK
    ctx = step.ctx.clone()
    ctx[0] = 16 * bt.shape[1] + 1  # longer than its table row
    status.zero_()
    pa.pa_decode(out, step.vals["q_decode"], step.kc, step.vc, step.bt, ctx, w.scale,
                 int(ctx.max()), device_status=status)
    assert int(status.item()) & pa.DEVFLAG_BAD_CONTEXT
    slots = torch.tensor([w.num_blocks * 16], dtype=torch.int64, device="cuda")
    status.zero_()
    k = torch.zeros(1, 8, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_reshape_and_cache(k, k, slots, step.kc, step.vc, device_status=status)
    assert int(status.item()) & pa.DEVFLAG_BAD_SLOT
    # the context stays usable
    assert torch.isfinite(step.decode().float()).all()


def test_workspace_too_small_is_rejected():
    w = wl.random_small(11, num_seqs=3, max_ctx=100)
    step = GpuStep(w)
    ws = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedKVError) as e:
        pa.pa_decode(torch.empty_like(step.vals["q_decode"]), step.vals["q_decode"], step.kc,
                     step.vc, step.bt, step.ctx, w.scale, 100, workspace=ws)
    assert e.value.status == pa.PA_ERR_WORKSPACE


def test_group_sizes_one_and_two():
    """GQA with 1 (plain MHA) and 2 query heads per kv head, against SDPA in float64."""
    for hq, hkv in ((8, 8), (16, 8)):
        rng = np.random.default_rng(hq)
        L = 77
        nb = 12
        table = rng.permutation(nb)[:5].astype(np.int32)[None]
        k = torch.randn(L, hkv, 64, device="cuda").to(torch.bfloat16)
        v = torch.randn(L, hkv, 64, device="cuda").to(torch.bfloat16)
        q = torch.randn(1, hq, 64, device="cuda").to(torch.bfloat16)
        kc = torch.full((nb, hkv, 16, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
        vc = kc.clone()
        bt = i32(table)
        ctx = i32([L])
        slots = pa.pa_compute_slot_mapping(bt, ctx, i32([0, L]), L, kc)
        pa.pa_reshape_and_cache(k, v, slots, kc, vc)
        out = torch.empty_like(q)
        pa.pa_decode(out, q, kc, vc, bt, ctx, 0.125, L)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.double().cpu()[:, :, None, :], k.double().cpu().transpose(0, 1)[None],
            v.double().cpu().transpose(0, 1)[None], scale=0.125, enable_gqa=True)[0, :, 0, :]
        mx, mean = errors(out.float().cpu().numpy()[0], ref.numpy())
        assert mx <= ATOL_MAX and mean <= ATOL_MEAN


@pytest.mark.parametrize("hq", [8, 16])
@pytest.mark.parametrize("partition_tokens", [0, 64])
def test_group_sizes_one_and_two_batched(hq, partition_tokens):
    """Group sizes 1 (8 query heads) and 2 (16) over a ragged batch of 12 sequences: the
    tensor-core tile arithmetic with 1 or 2 live MMA rows, runs split across sequences and
    merged in the attention kernel (balanced) or by the merge kernel (64-token partitions);
    pools bit-exact and outputs against the oracle."""
    w = wl.random_small(300 + hq + partition_tokens, num_seqs=12, max_ctx=900, num_q_heads=hq)
    full_check(w, partition_tokens=partition_tokens)


@pytest.mark.parametrize("partition_tokens", [0, 16, 512])
def test_group_sizes_one_and_two_long_context(partition_tokens):
    """Group sizes 1 and 2 over a 1500-token context: split segments merged in the attention
    kernel (balanced runs) or, with partitions, by the merge kernel's GROUP 1 and 2 forms
    (94 one-tile partials at 16 tokens), against SDPA in float64."""
    for hq, hkv in ((8, 8), (16, 8)):
        rng = np.random.default_rng(hq + partition_tokens)
        L = 1500
        nb = 110
        table = rng.permutation(nb)[:94].astype(np.int32)[None]
        k = torch.randn(L, hkv, 64, device="cuda").to(torch.bfloat16)
        v = torch.randn(L, hkv, 64, device="cuda").to(torch.bfloat16)
        q = torch.randn(1, hq, 64, device="cuda").to(torch.bfloat16)
        kc = torch.full((nb, hkv, 16, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
        vc = kc.clone()
        bt = i32(table)
        ctx = i32([L])
        status = pa.new_device_status()
        slots = pa.pa_compute_slot_mapping(bt, ctx, i32([0, L]), L, kc, device_status=status)
        pa.pa_reshape_and_cache(k, v, slots, kc, vc, device_status=status)
        out = torch.empty_like(q)
        pa.pa_decode(out, q, kc, vc, bt, ctx, 0.125, L, partition_tokens, device_status=status)
        assert pa.pa_check_device_status(status) == pa.PA_OK
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.double().cpu()[:, :, None, :], k.double().cpu().transpose(0, 1)[None],
            v.double().cpu().transpose(0, 1)[None], scale=0.125, enable_gqa=True)[0, :, 0, :]
        mx, mean = errors(out.float().cpu().numpy()[0], ref.numpy())
        assert mx <= ATOL_MAX and mean <= ATOL_MEAN, (hq, hkv, partition_tokens, mx, mean)


def test_split_segments_merged_in_kernel_and_workspace_reuse():
    """Contexts up to 8192 tokens are split over many warps and merged inside the attention
    kernel through per-segment counters; a reused workspace must give the same result."""
    w = wl.make_workload("long4", [7999, 7999, 6000, 4095], [1, 1, 1, 1], seed=12,
                         pool_slack=0.1)
    step = GpuStep(w)
    need = pa.pa_decode_workspace_size(4, 8, 32, int(w.context_lens.max()), 0)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        out = torch.empty_like(step.vals["q_decode"])
        pa.pa_decode(out, step.vals["q_decode"], step.kc, step.vc, step.bt, step.ctx, w.scale,
                     int(w.context_lens.max()), workspace=ws, device_status=step.status)
        outs.append(out)
    assert step.check_status() == pa.PA_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = oracle_step(w, host_vals(step.vals))
    assert_close(outs[0], ref["decode"], "long contexts, in-kernel merge")


@pytest.mark.parametrize("partition_tokens", [16, 32])
def test_merge_kernel_many_partials_and_workspace_reuse(partition_tokens):
    """Short partitions of contexts up to 3000 tokens give segments of up to about 190
    partials, and more runs than tiles (empty runs) for partitions of one tile; the merge
    kernel combines them, and a reused workspace must give the same result."""
    w = wl.make_workload("merge2", [2999, 40, 1777, 3000, 700, 1], [1, 1, 1, 1, 1, 1], seed=21,
                         pool_slack=0.1)
    step = GpuStep(w)
    mx = int(w.context_lens.max())
    need = pa.pa_decode_workspace_size(6, 8, 32, mx, partition_tokens)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        out = torch.empty_like(step.vals["q_decode"])
        pa.pa_decode(out, step.vals["q_decode"], step.kc, step.vc, step.bt, step.ctx, w.scale,
                     mx, partition_tokens, workspace=ws, device_status=step.status)
        outs.append(out)
    assert step.check_status() == pa.PA_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = oracle_step(w, host_vals(step.vals))
    assert_close(outs[0], ref["decode"], f"merge kernel, partitions of {partition_tokens}")


def test_a_wait_that_runs_out_reports_timeout_and_leaves_the_context_usable():
    status = pa.new_device_status()
    pa.pa_selftest_wait_timeout(status, limit_ms=50)
    assert pa.pa_check_device_status(status) == pa.PA_ERR_DEVICE_TIMEOUT
    assert int(status.item()) & pa.DEVFLAG_TIMEOUT
    w = wl.random_small(77, num_seqs=2, max_ctx=50)
    step = GpuStep(w)
    assert torch.isfinite(step.decode().float()).all()


def test_the_largest_batch_one_call_accepts():
    """4096 sequences (the per-call maximum) of 1..80 tokens: every (sequence, head) row,
    stores bit-exact; 4097 is refused on the host."""
    rng = np.random.default_rng(77)
    ctx = rng.integers(1, 81, size=4096)
    w = wl.make_workload("max_batch", ctx - 1, np.ones_like(ctx), seed=77, pool_slack=0.05)
    full_check(w)
    step = GpuStep(wl.make_workload("over", [3] * 4097, [1] * 4097, seed=1, pool_slack=0.0))
    out = torch.empty_like(step.vals["q_decode"])
    with pytest.raises(pa.PagedKVError):
        pa.pa_decode(out, step.vals["q_decode"], step.kc, step.vc, step.bt, step.ctx, 0.125, 4)
