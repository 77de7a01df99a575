"""A decode step captured in a CUDA graph and replayed gives the same bits as eager calls,
and replays pick up new buffer contents (the captured addresses stay fixed)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import graphs
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep, i32

pytestmark = pytest.mark.gpu


def test_captured_decode_step_replays_bit_identically():
    w = wl.decode_batch64_uniform()
    step = GpuStep(w, store_new=False)
    max_ctx = int(w.context_lens.max())
    need = pa.pa_decode_workspace_size(w.num_seqs, 8, 32, max_ctx, 0)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    q = step.vals["q_decode"].clone()
    out = torch.empty_like(q)

    def one_step():
        pa.pa_decode_append(out, q, step.vals["new_k"], step.vals["new_v"], step.kc, step.vc,
                            step.bt, step.ctx, w.scale, max_ctx, workspace=ws)

    cache = graphs.GraphCache(lambda batch: one_step)
    cache.run(w.num_seqs)
    torch.cuda.synchronize()
    replayed = out.clone()
    eager = torch.empty_like(out)
    pa.pa_decode_append(eager, q, step.vals["new_k"], step.vals["new_v"], step.kc, step.vc,
                        step.bt, step.ctx, w.scale, max_ctx, workspace=ws)
    assert torch.equal(replayed, eager)
    # new query contents, same buffers: the replay must see them
    q.copy_(torch.flip(step.vals["q_decode"], dims=[0]))
    cache.run(w.num_seqs)
    pa.pa_decode_append(eager, q, step.vals["new_k"], step.vals["new_v"], step.kc, step.vc,
                        step.bt, step.ctx, w.scale, max_ctx, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, eager) and not torch.equal(out, replayed)
    assert len(cache) == 1


def test_captured_prefill_and_decode_step():
    w = wl.make_workload("mix", [100, 37, 500, 20], [64, 40, 1, 1], num_prefill=2, seed=4,
                         pool_slack=0.3)
    step = GpuStep(w)
    out_p = torch.empty_like(step.vals["q_prefill"])
    out_d = torch.empty_like(step.vals["q_decode"])
    qsl = i32(w.prefill_query_start_loc)
    bt_p, ctx_p = step.bt[:2].contiguous(), step.ctx[:2].contiguous()
    bt_d, ctx_d = step.bt[2:].contiguous(), step.ctx[2:].contiguous()
    ws = torch.zeros(pa.pa_decode_workspace_size(2, 8, 32, 501, 0), dtype=torch.uint8,
                     device="cuda")

    def one_step():
        pa.pa_prefill_chunk(out_p, step.vals["q_prefill"], qsl, 64, step.kc, step.vc, bt_p,
                            ctx_p, w.scale)
        pa.pa_decode(out_d, step.vals["q_decode"], step.kc, step.vc, bt_d, ctx_d, w.scale, 501,
                     workspace=ws)

    g = graphs.StepGraph(one_step)
    out_p.zero_()
    out_d.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref_p, ref_d = out_p.clone(), out_d.clone()
    one_step()
    torch.cuda.synchronize()
    assert torch.equal(ref_p, out_p) and torch.equal(ref_d, out_d)
    assert torch.count_nonzero(ref_p) > 0
