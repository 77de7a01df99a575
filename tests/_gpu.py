"""GPU-side helpers for the parity tests: run a workload through the C-ABI library, and run
the same workload through the oracle on the host.  The two share only the seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import workloads as wl
from _util import oracle_pools


def i32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


class GpuStep:
    """Device state of one workload layer: NaN-poisoned pools filled with the history
    through the library's slot mapping + store, then this step's tokens stored."""

    def __init__(self, w: wl.Workload, layer=0, vals=None, store_new=True):
        self.w = w
        self.vals = vals if vals is not None else w.values(layer, "cuda")
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        self.kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        self.vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        self.bt = i32(w.block_tables)
        self.ctx = i32(w.context_lens)
        self.status = pa.new_device_status()
        hist_total = int(w.hist_lens.sum())
        self.hist_slots = pa.pa_compute_slot_mapping(self.bt, i32(w.hist_lens),
                                                     i32(w.hist_start_loc), hist_total, self.kc,
                                                     device_status=self.status)
        pa.pa_reshape_and_cache(self.vals["hist_k"], self.vals["hist_v"], self.hist_slots,
                                self.kc, self.vc, device_status=self.status)
        self.new_slots = None
        if store_new:
            self.store_new()

    def store_new(self):
        w = self.w
        self.new_slots = pa.pa_compute_slot_mapping(self.bt, self.ctx, i32(w.new_start_loc),
                                                    int(w.new_lens.sum()), self.kc,
                                                    device_status=self.status)
        pa.pa_reshape_and_cache(self.vals["new_k"], self.vals["new_v"], self.new_slots,
                                self.kc, self.vc, device_status=self.status)

    def decode(self, partition_tokens=None):
        w = self.w
        if partition_tokens is None:
            partition_tokens = w.partition_tokens
        out = torch.empty_like(self.vals["q_decode"])
        dctx = w.decode_context_lens
        pa.pa_decode(out, self.vals["q_decode"], self.kc, self.vc,
                     self.bt[w.num_prefill:].contiguous(), self.ctx[w.num_prefill:].contiguous(),
                     w.scale, int(dctx.max()) if len(dctx) else 0, partition_tokens,
                     device_status=self.status)
        return out

    def prefill(self):
        w = self.w
        out = torch.empty_like(self.vals["q_prefill"])
        qsl = w.prefill_query_start_loc
        pa.pa_prefill_chunk(out, self.vals["q_prefill"], i32(qsl),
                            int(w.new_lens[: w.num_prefill].max()), self.kc, self.vc,
                            self.bt[: w.num_prefill].contiguous(),
                            self.ctx[: w.num_prefill].contiguous(), w.scale,
                            device_status=self.status)
        return out

    def check_status(self):
        return pa.pa_check_device_status(self.status)


def host_vals(vals):
    return {k: v.to("cpu") for k, v in vals.items()}


def oracle_step(w: wl.Workload, hvals: dict):
    """Oracle pools and outputs for the same workload (host, double precision)."""
    kc, vc = oracle_pools(w, hvals)
    res = {"kc": kc, "vc": vc}
    if w.num_decode:
        res["decode"], err = oracle.decode(wl.bf16_bits(hvals["q_decode"]), kc, vc,
                                           w.decode_block_tables, w.decode_context_lens,
                                           w.scale)
        assert err == 0
    if w.num_prefill:
        res["prefill"], err = oracle.prefill_chunk(
            wl.bf16_bits(hvals["q_prefill"]), w.prefill_query_start_loc, kc, vc,
            w.block_tables[: w.num_prefill], w.context_lens[: w.num_prefill], w.scale)
        assert err == 0
    return res


def bits(t: torch.Tensor) -> np.ndarray:
    return wl.bf16_bits(t)
