"""The decode entry point that takes no workspace (pa_decode_static_scratch).

It serves callers that cannot allocate device memory, for example a plug-in whose host
program owns every device allocation, or code that must not call cudaMalloc while
serving because that call can stall the device.  The tests call it through the C ABI and
compare it with pa_decode (the entry point that takes a caller workspace) and with the
oracle, on calls in a row: two balanced-split calls of different batch sizes whose split
sequences are merged inside the kernel (the second runs on the array the first one
filled: where its piece counters sit depends on the batch size, so each call clears
them), then a fixed-partition call.  This file sorts last so that a
run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep, host_vals, oracle_step
from _util import ATOL_MAX, ATOL_MEAN, errors

pytestmark = pytest.mark.gpu


def _static_decode(step, partition_tokens):
    w = step.w
    out = torch.full_like(step.vals["q_decode"], float("nan"))
    status = pa.new_device_status()
    pa.pa_decode_static_scratch(out, step.vals["q_decode"], step.kc, step.vc,
                                step.bt[w.num_prefill:].contiguous(),
                                step.ctx[w.num_prefill:].contiguous(), w.scale,
                                int(w.decode_context_lens.max()), partition_tokens,
                                device_status=status)
    assert pa.pa_check_device_status(status) == pa.PA_OK
    return out


def _check(got, want, what):
    got = got.float().cpu().numpy().astype(np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.isfinite(got).all(), what
    mx, mean = errors(got, want)
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN, (what, mx, mean)


def test_static_scratch_matches_workspace_decode_and_oracle_on_calls_in_a_row():
    a = GpuStep(wl.decode_batch64_uniform())                   # 64 sequences, in-kernel merge
    b = GpuStep(wl.random_small(17, num_seqs=9, max_ctx=700))  # ragged, in-kernel merge
    outs = [(a, 0, _static_decode(a, 0)),
            (b, 0, _static_decode(b, 0)),     # counters where call 1 wrote offsets
            (b, 64, _static_decode(b, 64))]   # fixed 64-token runs, separate merge kernel
    torch.cuda.synchronize()
    refs = {id(s): oracle_step(s.w, host_vals(s.vals))["decode"] for s in (a, b)}
    for step, part, out in outs:
        _check(out, step.decode(part).float().cpu().numpy(), (step.w.name, part, "pa_decode"))
        _check(out, refs[id(step)], (step.w.name, part, "oracle"))


def test_balanced_split_of_the_largest_batch_fits_the_scratch_on_this_device():
    """A balanced split (partition_tokens 0) of the largest batch one call accepts (4096
    sequences, 8 K/V heads, 32 query heads, 8192-token contexts) fits the built-in array."""
    assert pa.PA_DECODE_STATIC_SCRATCH_BYTES == 8 << 20
    need = pa.pa_decode_workspace_size(4096, 8, 32, 8192, 0)
    assert 0 < need <= pa.PA_DECODE_STATIC_SCRATCH_BYTES


def test_sizes_beyond_the_scratch_are_rejected_before_launch():
    step = GpuStep(wl.make_workload("tiny", [20, 30], [1, 1], seed=3, pool_slack=0.5))
    need = pa.pa_decode_workspace_size(4, 8, 32, 131072, 256)  # 131072-token contexts
    assert need > pa.PA_DECODE_STATIC_SCRATCH_BYTES
    q = torch.zeros(4, 32, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 3.0)
    bt = torch.zeros(4, 8192, dtype=torch.int32, device="cuda")
    ctx = torch.full((4,), 131072, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedKVError) as e:
        pa.pa_decode_static_scratch(out, q, step.kc, step.vc, bt, ctx, 0.125, 131072, 256)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)  # nothing ran
