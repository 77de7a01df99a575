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
    kc = wl.nan_pool(w.num_blocks, w.num_kv_heads)
    vc = wl.nan_pool(w.num_blocks, w.num_kv_heads)
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


def oracle_prefill_rows(q_bits, query_start_loc, key_cache, value_cache, block_tables,
                        context_lens, scale, rows_per_task=128):
    """The oracle's causal chunk attention (pko_prefill_chunk) of every row, with the rows
    split into ranges that run on all host threads (ctypes releases the GIL during each
    call; the oracle keeps no shared state).  Rows [a, b) of a chunk of q_len rows over L
    keys are themselves the chunk of b - a rows over the first L - q_len + b keys: row i
    sits at position L - q_len + i either way.  Returns float64 [rows, Hq, D]."""
    import concurrent.futures as cf

    qsl = np.asarray(query_start_loc, dtype=np.int64)
    ctx = np.asarray(context_lens, dtype=np.int64)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    out = np.zeros(q_bits.shape, dtype=np.float64)
    tasks = []
    for s in range(len(qsl) - 1):
        q0, q1 = int(qsl[s]), int(qsl[s + 1])
        q_len, L = q1 - q0, int(ctx[s])
        for a in range(0, q_len, rows_per_task):
            b = min(q_len, a + rows_per_task)
            tasks.append((s, q0 + a, q0 + b, L - q_len + b))

    def run(task):
        s, r0, r1, keys = task
        o, err = oracle.prefill_chunk(q_bits[r0:r1], np.array([0, r1 - r0], np.int32),
                                      key_cache, value_cache, tables[s:s + 1],
                                      np.array([keys], np.int32), scale)
        assert err == 0, task
        out[r0:r1] = o

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(run, tasks))
    return out


def oracle_decode_rows(q_bits, key_cache, value_cache, block_tables, context_lens, scale,
                       seqs_per_task=8):
    """The oracle's decode attention (pko_decode) of every sequence, slices of sequences
    run on all host threads.  Returns float64 [S, Hq, D]."""
    import concurrent.futures as cf

    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros(q_bits.shape, dtype=np.float64)

    def run(a):
        b = min(len(ctx), a + seqs_per_task)
        o, err = oracle.decode(q_bits[a:b], key_cache, value_cache, tables[a:b], ctx[a:b],
                               scale)
        assert err == 0, a
        out[a:b] = o

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(run, range(0, len(ctx), seqs_per_task)))
    return out
