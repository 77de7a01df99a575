"""Helpers shared by the tests: golden-file parsing, oracle pool construction and the
dense (contiguous, logical-order) K/V view used by the library-routine checks."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from paged_kv_cache_299_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Attention tolerance for a bf16-output kernel against the double-precision oracle
# (bf16 in, fp32 accumulate): max-abs 2e-2, mean-abs 2e-3.
ATOL_MAX = 2e-2
ATOL_MEAN = 2e-3


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def oracle_pools(w: wl.Workload, vals: dict, include_new=True):
    """Build the oracle's own K/V pools: NaN-poisoned, history stored, then (optionally)
    this step's new tokens, each through the oracle's slot mapping and scatter."""
    kc = wl.nan_pool(w.num_blocks)
    vc = wl.nan_pool(w.num_blocks)
    hist_ctx = w.hist_lens
    slots, err = oracle.slot_mapping(w.block_tables, hist_ctx, w.hist_start_loc, w.num_blocks)
    assert err == 0
    assert oracle.reshape_and_cache(wl.bf16_bits(vals["hist_k"]), wl.bf16_bits(vals["hist_v"]),
                                    slots, kc, vc) == 0
    if include_new:
        slots, err = oracle.slot_mapping(w.block_tables, w.context_lens, w.new_start_loc,
                                         w.num_blocks)
        assert err == 0
        assert oracle.reshape_and_cache(wl.bf16_bits(vals["new_k"]),
                                        wl.bf16_bits(vals["new_v"]), slots, kc, vc) == 0
    return kc, vc


def dense_kv(w: wl.Workload, vals: dict, s: int):
    """Sequence s's keys and values in logical order, float64 [Hkv, L, D]: its history
    followed by its new tokens (no paging involved)."""
    hs, he = w.hist_start_loc[s], w.hist_start_loc[s + 1]
    ns, ne = w.new_start_loc[s], w.new_start_loc[s + 1]
    k = torch.cat([vals["hist_k"][hs:he], vals["new_k"][ns:ne]]).to(torch.float64)
    v = torch.cat([vals["hist_v"][hs:he], vals["new_v"][ns:ne]]).to(torch.float64)
    return k.transpose(0, 1).contiguous(), v.transpose(0, 1).contiguous()


def sdpa_decode(w: wl.Workload, vals: dict, s_dec: int):
    """torch scaled_dot_product_attention (float64, CPU) of decode sequence s_dec's query
    over its dense K/V, GQA through enable_gqa.  Returns [Hq, D]."""
    s = w.num_prefill + s_dec
    k, v = dense_kv(w, vals, s)
    q = vals["q_decode"][s_dec].to(torch.float64)[:, None, :]  # [Hq, 1, D]
    o = torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None], v[None], scale=w.scale, enable_gqa=True)
    return o[0, :, 0, :]


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = np.abs(got - ref)
    return float(diff.max()) if diff.size else 0.0, float(diff.mean()) if diff.size else 0.0
