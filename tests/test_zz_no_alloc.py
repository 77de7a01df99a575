"""The decode entry point that takes no workspace (pa_decode_static_scratch).

It serves callers that cannot allocate device memory, for example a plug-in whose host
program owns every device allocation, or code that must not call cudaMalloc while
serving because that call can stall the device.  The tests call it through the C ABI
and compare it with pa_decode (the entry point that takes a caller workspace) on two
calls in a row, so the second call runs on scratch the first one left behind.  This file
sorts last so that a run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep
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


def test_static_scratch_matches_workspace_decode_on_two_calls_in_a_row():
    a = GpuStep(wl.decode_batch64_uniform())                                  # 64 sequences, balanced split
    b = GpuStep(wl.random_small(17, num_seqs=9, max_ctx=700))  # ragged, fixed 64-token runs
    out_a = _static_decode(a, 0)
    out_b = _static_decode(b, 64)  # second call: reuses the scratch the first one wrote
    torch.cuda.synchronize()
    for step, out, part in ((a, out_a, 0), (b, out_b, 64)):
        ref = step.decode(part)
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        mx, mean = errors(got, want)
        assert mx <= ATOL_MAX and mean <= ATOL_MEAN, (step.w.name, mx, mean)


def test_sizes_beyond_the_scratch_are_rejected_before_launch():
    step = GpuStep(wl.make_workload("tiny", [20, 30], [1, 1], seed=3, pool_slack=0.5))
    need = pa.pa_decode_workspace_size(4, 8, 32, 131072, 512)  # 131072-token contexts, 512 runs
    assert need > 4 << 20
    q = torch.zeros(4, 32, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 3.0)
    bt = torch.zeros(4, 8192, dtype=torch.int32, device="cuda")
    ctx = torch.full((4,), 131072, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedKVError) as e:
        pa.pa_decode_static_scratch(out, q, step.kc, step.vc, bt, ctx, 0.125, 131072, 512)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)  # nothing ran
