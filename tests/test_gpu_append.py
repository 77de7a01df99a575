"""pa_decode_append (store of the newest token fused into decode) must be bit-identical to
pa_reshape_and_cache followed by pa_decode: same pools, same outputs."""
import numpy as np
import pytest
import torch

from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep, host_vals, i32, oracle_step
from _util import ATOL_MAX, ATOL_MEAN, errors

pytestmark = pytest.mark.gpu


def both_paths(w, layer=0, partition_tokens=0):
    step = GpuStep(w, layer, store_new=False)  # history only
    kc2, vc2 = step.kc.clone(), step.vc.clone()
    max_ctx = int(w.context_lens.max())
    # separate: slot mapping + store, then decode
    step.store_new()
    out_a = torch.empty_like(step.vals["q_decode"])
    pa.pa_decode(out_a, step.vals["q_decode"], step.kc, step.vc, step.bt, step.ctx, w.scale,
                 max_ctx, partition_tokens, device_status=step.status)
    # fused
    out_b = torch.empty_like(out_a)
    pa.pa_decode_append(out_b, step.vals["q_decode"], step.vals["new_k"], step.vals["new_v"],
                        kc2, vc2, step.bt, step.ctx, w.scale, max_ctx, partition_tokens,
                        device_status=step.status)
    assert step.check_status() == pa.PA_OK
    assert torch.equal(step.kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(step.vc.view(torch.int16), vc2.view(torch.int16))
    assert torch.equal(out_a, out_b)
    return step, out_b


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fused_append_equals_store_then_decode_small(seed):
    both_paths(wl.random_small(200 + seed, num_seqs=7, max_ctx=400))


@pytest.mark.parametrize("partition_tokens", [0, 16, 512])
def test_fused_append_all_tail_lengths(partition_tokens):
    ctx = np.arange(1, 81)
    w = wl.make_workload("tails", ctx - 1, np.ones_like(ctx), seed=9, pool_slack=0.25)
    both_paths(w, partition_tokens=partition_tokens)


def test_fused_append_decode_batch64_against_oracle():
    w = wl.decode_batch64_uniform()
    step, out = both_paths(w)
    ref = oracle_step(w, host_vals(step.vals))
    mx, mean = errors(out.float().cpu().numpy(), ref["decode"])
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN


def test_fused_append_batch256_layer():
    both_paths(wl.decode_batch256_lognormal(layers=1))
