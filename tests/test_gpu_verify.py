"""Speculative-decoding verification ("vLLM", Speculative Decoding: the target model checks
K drafted tokens in one pass): the K+1 positions (newest accepted token + K drafts) are a
causal chunk over the paged prefix, so pa_prefill_chunk scores them in one launch.  Each
row must equal decode over its own prefix (oracle), for every K and prefix length."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _gpu import GpuStep, host_vals
from _util import ATOL_MAX, ATOL_MEAN, errors, oracle_pools

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("k_draft", [1, 3, 4, 7])
def test_verify_rows_equal_decode_over_each_prefix(k_draft):
    prefixes = [15, 16, 129, 1000, 2047, 5]
    q_len = k_draft + 1
    w = wl.make_workload(f"verify{k_draft}", prefixes, [q_len] * len(prefixes),
                         num_prefill=len(prefixes), seed=30 + k_draft, pool_slack=0.2)
    step = GpuStep(w)
    out = step.prefill()
    assert step.check_status() == pa.PA_OK
    hv = host_vals(step.vals)
    kc, vc = oracle_pools(w, hv)
    qsl = w.prefill_query_start_loc
    rows, ctx, tables = [], [], []
    for s, p in enumerate(prefixes):
        for i in range(q_len):  # draft i sees the prefix and drafts 0..i
            rows.append(qsl[s] + i)
            ctx.append(p + i + 1)
            tables.append(w.block_tables[s])
    ref, err = oracle.decode(wl.bf16_bits(hv["q_prefill"])[rows], kc, vc, np.stack(tables),
                             np.array(ctx, np.int32), w.scale)
    assert err == 0
    mx, mean = errors(out[torch.tensor(rows, device="cuda")].float().cpu().numpy(), ref)
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN, (mx, mean)
