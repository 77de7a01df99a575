"""Unified varlen launch ("vLLM", Continuous Batching: decode rows and prefill chunks of
different sequences share one step): pa_attention_varlen over a mixed batch must equal the
oracle's causal chunk attention for every row (a q_len = 1 sequence is a decode row),
whatever the order of the sequences; its chunk rows come from the tensor-core kernel and
are bit-identical to pa_prefill_chunk, its decode rows from the decode kernel."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep, host_vals, i32
from _util import (ATOL_MAX, ATOL_MEAN, errors, oracle_decode_rows, oracle_pools,
                   oracle_prefill_rows)

pytestmark = pytest.mark.gpu


def permuted(step, order):
    """q rows, query_start_loc, block tables and context lengths of the step's sequences
    taken in `order`."""
    w = step.w
    qsl = w.prefill_query_start_loc
    segs = [step.vals["q_prefill"][qsl[s]:qsl[s + 1]] for s in order]
    q = torch.cat(segs).contiguous()
    lens = np.array([qsl[s + 1] - qsl[s] for s in order], np.int32)
    qsl2 = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx = torch.tensor(order, device="cuda", dtype=torch.long)
    return q, qsl2, step.bt[idx].contiguous(), step.ctx[idx].contiguous(), lens


def check(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    mx, mean = errors(g, ref)
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN, f"{what}: max {mx:.3g} mean {mean:.3g}"


@pytest.mark.parametrize("seed", range(5))
def test_mixed_batch_any_order_matches_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    n = 12
    hist = rng.integers(0, 700, size=n)
    new = np.where(rng.random(n) < 0.6, 1, rng.integers(2, 150, size=n))  # mostly decode rows
    w = wl.make_workload(f"varlen{seed}", hist, new, num_prefill=n, seed=200 + seed,
                         pool_slack=0.3)
    step = GpuStep(w)
    order = rng.permutation(n)
    q, qsl, bt, ctx, lens = permuted(step, order)
    out = torch.empty_like(q)
    pa.pa_attention_varlen(out, q, i32(qsl), int(lens.max()), step.kc, step.vc, bt, ctx,
                           w.scale, device_status=step.status)
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref, err = oracle.prefill_chunk(wl.bf16_bits(q.cpu()), qsl, kc, vc, bt.cpu().numpy(),
                                    ctx.cpu().numpy(), w.scale)
    assert err == 0
    check(out, ref, w.name)
    # chunk rows come from the same tensor-core kernel as pa_prefill_chunk: bit-identical;
    # decode rows (q_len 1) from the CUDA-core decode kernel: equal within rounding
    same = torch.empty_like(q)
    pa.pa_prefill_chunk(same, q, i32(qsl), int(lens.max()), step.kc, step.vc, bt, ctx, w.scale)
    one = torch.from_numpy(np.repeat(lens == 1, lens)).cuda()
    assert torch.equal(out[~one], same[~one])
    assert (out[one].float() - same[one].float()).abs().max().item() <= 1.6e-2


def test_mixed_step_matches_chunk_and_decode_kernels_and_oracle():
    """The mixed continuous-batching step (8 chunks of 512 and 248 decode rows) in one
    varlen call: its chunk rows equal pa_prefill_chunk bit for bit, its decode rows agree
    with pa_decode within the attention tolerance, and every row matches the oracle."""
    w = wl.mixed_prefill_decode()
    step = GpuStep(w)
    nd = w.num_decode
    qsl_pre = w.prefill_query_start_loc
    tp = int(qsl_pre[-1])
    qsl = np.concatenate([qsl_pre, tp + np.arange(1, nd + 1)]).astype(np.int32)
    q = torch.cat([step.vals["q_prefill"], step.vals["q_decode"]]).contiguous()
    out = torch.empty_like(q)
    ws = torch.empty(pa.pa_varlen_workspace_size(w.num_seqs, q.shape[0]), dtype=torch.uint8,
                     device="cuda")
    for _ in range(2):  # the workspace needs no clearing between calls
        pa.pa_attention_varlen(out, q, i32(qsl), 512, step.kc, step.vc, step.bt, step.ctx,
                               w.scale, workspace=ws, device_status=step.status)
    assert step.check_status() == pa.PA_OK
    same = torch.empty_like(q)
    pa.pa_prefill_chunk(same, q, i32(qsl), 512, step.kc, step.vc, step.bt, step.ctx, w.scale)
    assert torch.equal(out[:tp], same[:tp])
    dec = step.decode()
    assert (out[tp:].float() - dec.float()).abs().max().item() <= 1.6e-2
    # every row of the step against the oracle: the 4096 chunk rows (causal chunks) and the
    # 248 decode rows (one query over the whole context)
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref_pre = oracle_prefill_rows(wl.bf16_bits(hv["q_prefill"]), qsl_pre, kc, vc,
                                  w.block_tables[: w.num_prefill],
                                  w.context_lens[: w.num_prefill], w.scale)
    ref_dec = oracle_decode_rows(wl.bf16_bits(hv["q_decode"]), kc, vc, w.decode_block_tables,
                                 w.decode_context_lens, w.scale)
    check(out, np.concatenate([ref_pre, ref_dec]), "mixed step, every row")


def test_mixed_step_with_the_decode_rows_beside_the_chunks():
    """The same mixed step with PA_LAUNCH_MAX_SMS: the decode rows on part of the SMs, the
    chunks on the others at the same time.  Chunk rows stay bit-identical to
    pa_prefill_chunk, decode rows match the oracle, and unknown flags are refused."""
    w = wl.mixed_prefill_decode()
    step = GpuStep(w)
    nd = w.num_decode
    qsl_pre = w.prefill_query_start_loc
    tp = int(qsl_pre[-1])
    qsl = np.concatenate([qsl_pre, tp + np.arange(1, nd + 1)]).astype(np.int32)
    q = torch.cat([step.vals["q_prefill"], step.vals["q_decode"]]).contiguous()
    ws = torch.empty(pa.pa_varlen_workspace_size(w.num_seqs, q.shape[0]), dtype=torch.uint8,
                     device="cuda")
    same = torch.empty_like(q)
    pa.pa_prefill_chunk(same, q, i32(qsl), 512, step.kc, step.vc, step.bt, step.ctx, w.scale)
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref_dec = oracle_decode_rows(wl.bf16_bits(hv["q_decode"]), kc, vc, w.decode_block_tables,
                                 w.decode_context_lens, w.scale)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for d in (2, sms // 2 + 14, sms + 10):  # the last one: the default schedule
        out = torch.full_like(q, float("nan"))
        for _ in range(2):
            pa.pa_attention_varlen(out, q, i32(qsl), 512, step.kc, step.vc, step.bt, step.ctx,
                                   w.scale, workspace=ws, device_status=step.status,
                                   launch_flags=pa.PA_LAUNCH_MAX_SMS(d))
        torch.cuda.synchronize()
        assert step.check_status() == pa.PA_OK
        assert torch.equal(out[:tp], same[:tp]), d
        check(out[tp:], ref_dec, f"decode rows on {d} SMs")
    with pytest.raises(pa.PagedKVError) as e:
        pa.pa_attention_varlen(out, q, i32(qsl), 512, step.kc, step.vc, step.bt, step.ctx,
                               w.scale, workspace=ws,
                               launch_flags=pa.PA_LAUNCH_OVERLAP_PREVIOUS)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


def test_empty_sequences_and_one_long_chunk():
    """q_len 0 sequences contribute nothing; a 700-row chunk (22 tiles) among decode rows."""
    hist = [40, 0, 300, 25, 1000, 7]
    new = [1, 700, 1, 1, 1, 3]
    w = wl.make_workload("varlen_edge", hist, new, num_prefill=6, seed=9, pool_slack=0.3)
    step = GpuStep(w)
    keep = [0, 1, 2, 4, 5]  # sequence 3 gets q_len 0 in the call (its row is dropped)
    qsl0 = w.prefill_query_start_loc
    q = torch.cat([step.vals["q_prefill"][qsl0[s]:qsl0[s + 1]] for s in keep]).contiguous()
    lens = np.array([qsl0[s + 1] - qsl0[s] if s in keep else 0 for s in range(6)], np.int32)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out = torch.empty_like(q)
    pa.pa_attention_varlen(out, q, i32(qsl), 700, step.kc, step.vc, step.bt, step.ctx,
                           w.scale, device_status=step.status)
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref, err = oracle.prefill_chunk(wl.bf16_bits(q.cpu()), qsl, kc, vc, w.block_tables,
                                    w.context_lens, w.scale)
    assert err == 0
    check(out, ref, "edge")


def test_rows_beyond_the_query_buffer_are_flagged_not_written():
    w = wl.make_workload("varlen_bad", [30, 50], [1, 20], num_prefill=2, seed=4, pool_slack=0.5)
    step = GpuStep(w)
    q = step.vals["q_prefill"]
    qsl = np.array([0, 1, 40], np.int32)  # the second sequence claims rows 1..39 of 21
    guard = torch.empty((64,) + tuple(q.shape[1:]), dtype=q.dtype, device="cuda")
    guard.fill_(3.0)
    out = guard[:q.shape[0]]
    status = pa.new_device_status()
    pa.pa_attention_varlen(out, q, i32(qsl), 20, step.kc, step.vc, step.bt, step.ctx, w.scale,
                           device_status=status)
    assert pa.pa_check_device_status(status) == pa.PA_ERR_DEVICE_INDEX
    assert torch.all(guard[q.shape[0]:] == 3.0)  # nothing written past the buffer
    assert torch.isfinite(out[0].float()).all()  # the valid sequence was still served


def test_decode_only_batch_runs_on_the_decode_kernel():
    """A batch of decode rows only (batch 256, lognormal contexts): every row comes from
    the CUDA-core decode kernel and equals pa_decode within rounding and the oracle."""
    w = wl.decode_batch256_lognormal(layers=1)
    step = GpuStep(w)
    q = step.vals["q_decode"]
    qsl = np.arange(w.num_seqs + 1, dtype=np.int32)
    out = torch.full_like(q, float("nan"))
    pa.pa_attention_varlen(out, q, i32(qsl), 1, step.kc, step.vc, step.bt, step.ctx, w.scale,
                           device_status=step.status)
    assert step.check_status() == pa.PA_OK
    dec = step.decode()
    assert (out.float() - dec.float()).abs().max().item() <= 1.6e-2
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref = oracle_decode_rows(wl.bf16_bits(hv["q_decode"]), kc, vc, w.block_tables,
                             w.context_lens, w.scale)
    check(out, ref, "decode-only varlen")


def test_more_sequences_than_the_decode_kernel_takes():
    """4100 one-row sequences (beyond the decode kernel's 4096): every row then runs on the
    tensor-core chunk kernel, in grid order (the batch is beyond the in-kernel sort too)."""
    rng = np.random.default_rng(41)
    ctx = rng.integers(1, 48, size=4100)
    w = wl.make_workload("many_rows", ctx - 1, np.ones(4100, np.int64), num_prefill=4100, seed=41,
                         pool_slack=0.2)
    step = GpuStep(w)
    q = step.vals["q_prefill"]
    out = torch.empty_like(q)
    pa.pa_attention_varlen(out, q, i32(w.prefill_query_start_loc), 1, step.kc, step.vc, step.bt,
                           step.ctx, w.scale, device_status=step.status)
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    ref = oracle_decode_rows(wl.bf16_bits(hv["q_prefill"]), kc, vc, w.block_tables,
                             w.context_lens, w.scale)
    check(out, ref, "4100 rows")
