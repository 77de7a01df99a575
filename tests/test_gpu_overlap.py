"""Decode launches that overlap the kernel before them (PA_LAUNCH_OVERLAP_PREVIOUS,
programmatic dependent launch).  A decode step over several layers, each layer with its
own pools and the launches after the first carrying the flag, must give the same bits as
the same step without the flag, eagerly and replayed from a CUDA graph, and must agree
with the oracle.  The layers share one workspace, so a launch that touched it before the
previous layer had finished would show up as wrong rows.  The mixed step's decode behind a
chunk prefill is checked the same way.  (The unified varlen launch starts its chunk kernel
behind its decode kernel in the same manner; its tests are in test_gpu_varlen.py.)"""
import pytest
import torch

from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import graphs
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep, host_vals, oracle_step
from _util import ATOL_MAX, ATOL_MEAN, errors

pytestmark = pytest.mark.gpu

LAYERS = 4


def _layers(w):
    # history only: every run below appends the step's token itself (an idempotent store)
    return [GpuStep(w, layer, store_new=False) for layer in range(LAYERS)]


def _run(steps, outs, ws, partition_tokens, overlap):
    w = steps[0].w
    max_ctx = int(w.context_lens.max())
    for i, st in enumerate(steps):
        flags = pa.PA_LAUNCH_OVERLAP_PREVIOUS if overlap and i > 0 else pa.PA_LAUNCH_DEFAULT
        pa.pa_decode_append(outs[i], st.vals["q_decode"], st.vals["new_k"], st.vals["new_v"],
                            st.kc, st.vc, st.bt, st.ctx, w.scale, max_ctx, partition_tokens,
                            workspace=ws, device_status=st.status, launch_flags=flags)


@pytest.mark.parametrize("name,partition_tokens", [("batch64", 0), ("small_merge", 64),
                                                   ("batch256", 0)])
def test_overlapped_layers_match_serial_layers_and_oracle(name, partition_tokens):
    w = {"batch64": lambda: wl.decode_batch64_uniform(),
         "small_merge": lambda: wl.random_small(41, num_seqs=9, max_ctx=900),
         "batch256": lambda: wl.decode_batch256_lognormal(layers=1)}[name]()
    steps = _layers(w)
    max_ctx = int(w.context_lens.max())
    ws = torch.zeros(max(16, pa.pa_decode_workspace_size(w.num_seqs, 8, 32, max_ctx,
                                                         partition_tokens)),
                     dtype=torch.uint8, device="cuda")
    serial = [torch.full_like(st.vals["q_decode"], float("nan")) for st in steps]
    overlapped = [torch.full_like(st.vals["q_decode"], float("nan")) for st in steps]
    _run(steps, serial, ws, partition_tokens, overlap=False)
    for _ in range(3):  # repeated steps: the start-up of one layer meets the tail of another
        _run(steps, overlapped, ws, partition_tokens, overlap=True)
        torch.cuda.synchronize()
        for a, b in zip(serial, overlapped):
            assert torch.equal(a, b)
    for st in steps:
        assert st.check_status() == pa.PA_OK
    for st, out in zip(steps, overlapped):
        ref = oracle_step(w, host_vals(st.vals))["decode"]
        mx, mean = errors(out.float().cpu().numpy(), ref)
        assert mx <= ATOL_MAX and mean <= ATOL_MEAN, (name, mx, mean)


def test_overlapped_layers_replay_from_a_graph():
    w = wl.decode_batch64_uniform()
    steps = _layers(w)
    max_ctx = int(w.context_lens.max())
    ws = torch.zeros(pa.pa_decode_workspace_size(w.num_seqs, 8, 32, max_ctx, 0),
                     dtype=torch.uint8, device="cuda")
    serial = [torch.empty_like(st.vals["q_decode"]) for st in steps]
    replayed = [torch.full_like(st.vals["q_decode"], float("nan")) for st in steps]
    _run(steps, serial, ws, 0, overlap=False)
    graph = graphs.StepGraph(lambda: _run(steps, replayed, ws, 0, overlap=True))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(serial, replayed):
        assert torch.equal(a, b)


def test_unknown_launch_flags_are_rejected():
    w = wl.random_small(5, num_seqs=2, max_ctx=40)
    st = GpuStep(w)
    out = torch.full_like(st.vals["q_decode"], 7.0)
    with pytest.raises(pa.PagedKVError) as e:
        pa.pa_decode(out, st.vals["q_decode"], st.kc, st.vc, st.bt, st.ctx, w.scale,
                     int(w.context_lens.max()), launch_flags=4)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing ran


def test_decode_behind_a_chunk_prefill_overlaps_it():
    """The mixed step: chunk prefill, then the decode of the one-token sequences with the
    flag (the prefill writes only its own output rows).  Both outputs match the serial
    launches bit for bit, and the decode rows match the oracle."""
    w = wl.mixed_prefill_decode()
    st = GpuStep(w)  # history and this step's tokens stored
    P = w.num_prefill
    qsl = torch.from_numpy(w.prefill_query_start_loc.astype("int32")).cuda()
    max_q = int(w.new_lens[:P].max())
    bt_p, ctx_p = st.bt[:P].contiguous(), st.ctx[:P].contiguous()
    bt_d, ctx_d = st.bt[P:].contiguous(), st.ctx[P:].contiguous()
    max_ctx = int(w.decode_context_lens.max())
    ws = torch.zeros(pa.pa_decode_workspace_size(w.num_decode, 8, 32, max_ctx, 0),
                     dtype=torch.uint8, device="cuda")

    def run(flags, out_p, out_d):
        pa.pa_prefill_chunk(out_p, st.vals["q_prefill"], qsl, max_q, st.kc, st.vc, bt_p, ctx_p,
                            w.scale, device_status=st.status)
        pa.pa_decode(out_d, st.vals["q_decode"], st.kc, st.vc, bt_d, ctx_d, w.scale, max_ctx,
                     workspace=ws, device_status=st.status, launch_flags=flags)

    serial_p = torch.empty_like(st.vals["q_prefill"])
    serial_d = torch.empty_like(st.vals["q_decode"])
    run(pa.PA_LAUNCH_DEFAULT, serial_p, serial_d)
    over_p = torch.full_like(serial_p, float("nan"))
    over_d = torch.full_like(serial_d, float("nan"))
    for _ in range(3):
        run(pa.PA_LAUNCH_OVERLAP_PREVIOUS, over_p, over_d)
    torch.cuda.synchronize()
    assert st.check_status() == pa.PA_OK
    assert torch.equal(serial_p, over_p) and torch.equal(serial_d, over_d)
    ref = oracle_step(w, host_vals(st.vals))["decode"]
    mx, mean = errors(over_d.float().cpu().numpy(), ref)
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN, (mx, mean)


@pytest.mark.parametrize("decode_share", [1, 40, "half", "all_but_one"])
def test_decode_beside_a_chunk_prefill_on_separate_sms(decode_share):
    """The mixed step with the decode confined to part of the SMs (PA_LAUNCH_MAX_SMS) and the
    chunk prefill launched right behind it on the other SMs (PA_LAUNCH_OVERLAP_PREVIOUS |
    PA_LAUNCH_MAX_SMS), so that both run at the same time: the chunk rows are bit-identical
    to the serial launches (a unit's arithmetic does not depend on the grid), the decode
    rows match the oracle (with fewer warps the split points move, so their rounding may
    differ from the serial decode's), eagerly and replayed from a CUDA graph."""
    w = wl.mixed_prefill_decode()
    st = GpuStep(w)
    P = w.num_prefill
    qsl = torch.from_numpy(w.prefill_query_start_loc.astype("int32")).cuda()
    max_q = int(w.new_lens[:P].max())
    bt_p, ctx_p = st.bt[:P].contiguous(), st.ctx[:P].contiguous()
    bt_d, ctx_d = st.bt[P:].contiguous(), st.ctx[P:].contiguous()
    max_ctx = int(w.decode_context_lens.max())
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    d = {1: 1, 40: 40, "half": sms // 2, "all_but_one": sms - 1}[decode_share]
    ws = torch.zeros(pa.pa_decode_workspace_size(w.num_decode, 8, 32, max_ctx, 0),
                     dtype=torch.uint8, device="cuda")
    serial_p = torch.empty_like(st.vals["q_prefill"])
    serial_d = torch.empty_like(st.vals["q_decode"])
    pa.pa_prefill_chunk(serial_p, st.vals["q_prefill"], qsl, max_q, st.kc, st.vc, bt_p, ctx_p,
                        w.scale, device_status=st.status)
    pa.pa_decode(serial_d, st.vals["q_decode"], st.kc, st.vc, bt_d, ctx_d, w.scale, max_ctx,
                 workspace=ws, device_status=st.status)

    def run(out_p, out_d):
        pa.pa_decode(out_d, st.vals["q_decode"], st.kc, st.vc, bt_d, ctx_d, w.scale, max_ctx,
                     workspace=ws, device_status=st.status, launch_flags=pa.PA_LAUNCH_MAX_SMS(d))
        pa.pa_prefill_chunk(out_p, st.vals["q_prefill"], qsl, max_q, st.kc, st.vc, bt_p, ctx_p,
                            w.scale, device_status=st.status,
                            launch_flags=pa.PA_LAUNCH_OVERLAP_PREVIOUS | pa.PA_LAUNCH_MAX_SMS(sms - d))

    conc_p = torch.full_like(serial_p, float("nan"))
    conc_d = torch.full_like(serial_d, float("nan"))
    for _ in range(2):
        run(conc_p, conc_d)
    torch.cuda.synchronize()
    assert st.check_status() == pa.PA_OK
    assert torch.equal(serial_p, conc_p)
    ref = oracle_step(w, host_vals(st.vals))["decode"]
    mx, mean = errors(conc_d.float().cpu().numpy(), ref)
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN, (d, mx, mean)
    graph_p = torch.full_like(serial_p, float("nan"))
    graph_d = torch.full_like(serial_d, float("nan"))
    graph = graphs.StepGraph(lambda: run(graph_p, graph_d))
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert st.check_status() == pa.PA_OK
    assert torch.equal(graph_p, serial_p) and torch.equal(graph_d, conc_d)


@pytest.mark.parametrize("decode_sms", [1, 50, 100])
def test_fixed_partitions_under_an_sm_budget_fit_the_size_query(decode_sms):
    """Fixed 512-token partitions of 64000 tokens give 1000 runs.  Under an SM budget with
    fewer warps than runs, rounding the runs up to a multiple of the budget's warp count
    would need more partials than the size query (which knows no budget) provides; the plan
    keeps the whole device's run count instead.  The call succeeds in exactly that
    workspace, reuses it, and matches the oracle."""
    w = wl.make_workload("budget", [15999, 15999, 14000, 9000], [1, 1, 1, 1], seed=31,
                         pool_slack=0.05)
    step = GpuStep(w)
    mx = int(w.context_lens.max())
    need = pa.pa_decode_workspace_size(4, 8, 32, mx, 512)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        out = torch.empty_like(step.vals["q_decode"])
        pa.pa_decode(out, step.vals["q_decode"], step.kc, step.vc, step.bt, step.ctx, w.scale,
                     mx, 512, workspace=ws, device_status=step.status,
                     launch_flags=pa.PA_LAUNCH_MAX_SMS(decode_sms))
        outs.append(out)
    assert step.check_status() == pa.PA_OK
    assert torch.equal(outs[0], outs[1])
    ref = oracle_step(w, host_vals(step.vals))["decode"]
    mxe, mean = errors(outs[0].float().cpu().numpy(), ref)
    assert mxe <= ATOL_MAX and mean <= ATOL_MEAN, (decode_sms, mxe, mean)
