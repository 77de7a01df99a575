#!/usr/bin/env python3
"""Benchmark of the paged KV-cache hot path on one GB300 (or N replicas under torchrun).

One step = one pass of the whole path over one batch: slot mapping of the step's new
tokens, then for every layer the KV store of the new tokens and paged attention (decode,
plus causal chunked prefill where the workload has chunks).  When every sequence adds one
token, the store rides in the decode launch (pa_decode_append), and the layers after the
first start under PA_LAUNCH_OVERLAP_PREVIOUS.  The default workload is decode batch 256
with lognormal contexts (median 1024, sigma 0.8, clipped to [1, 8192]) and 16 layers of
KV pools resident; other workloads are reachable with --workload.

Prints ONE JSON line (rank 0).  ``value`` is KV-read GB/s: the live K+V bytes the decode
attention must read in a step (sum of context lengths x 2048 B x layers), divided by the
device time of the whole step; tokens/s is batch / step time.

``--impl reference`` times the CPU oracle (plain C, double precision) on a bounded sample
of the same workload: the slow baseline arm, not a target.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn: KV-read HBM GB/s (% of GB300 peak); tokens/s at batch 256"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="decode_b256",
                    choices=["single_seq_300", "decode_b64", "decode_b256", "long_context_b4",
                             "mixed_step"])
    ap.add_argument("--mixed", choices=["split", "unified", "concurrent"], default="split",
                    help="steps with prefill chunks and decode rows: pa_prefill_chunk then "
                         "pa_decode; one pa_attention_varlen over all sequences; or the "
                         "decode on part of the SMs with the chunk prefill beside it")
    ap.add_argument("--append", choices=["fused", "separate"], default="fused",
                    help="decode-only steps: store the new tokens inside the decode launch "
                         "(pa_decode_append) or with pa_reshape_and_cache first")
    ap.add_argument("--launch", choices=["eager", "graph"], default="graph",
                    help="time the step as eager C-ABI calls or as one CUDA-graph replay")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernels-only", action="store_true",
                    help="time only the standalone store and copy-on-write kernels (a short "
                         "run for profilers) and print their figures")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other workloads and the standalone store measurement")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--flush", choices=["write-read", "write"], default="write-read",
                    help="L2 flush between steps of workloads smaller than 4x L2: rewrite a "
                         "2x L2 buffer, then read another (so the step starts from clean "
                         "lines), or only rewrite it")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (small cases for profilers)")
    return ap.parse_args()


def ncu_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch of `kernel` on `workload_key` from the committed ncu figures in
    profiles/dram_traffic.json, if they were taken with the kernel's current source (else
    None: the counters no longer describe the kernel that runs)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            entry = json.load(f)[kernel]
        with open(os.path.join(ROOT, entry["source"]), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
        if entry["source_sha256"] != digest:
            return None
        v = entry["workloads"].get(workload_key, {}).get("dram_bytes_per_launch")
        return int(v) if v else None
    except Exception:
        return None


def max_over_ranks(value: float, device) -> float:
    """Slowest rank's time (every rank gets it); identity for a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: int, world: int, step_ms: float) -> float:
    """Weak scaling: every rank moves bytes_per_rank per step; the job's throughput is
    all ranks' bytes over the slowest rank's step time."""
    return bytes_per_rank * world / (step_ms * 1e-3) / 1e9


def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The decode beside the chunk prefill (PA_LAUNCH_MAX_SMS): the decode's share of the SMs is
# chosen so that both end together, from per-SM rates measured on a GB300 (decode with one
# CTA per SM beside the prefill: about 61 GB/s of K/V per SM, 6.2 TB/s at most in all;
# chunk prefill: about 3.75 TFLOP/s of causal-useful work per SM at two CTAs per SM).
DECODE_GBS_PER_SM = 61.0
DECODE_GBS_MAX = 6200.0
PREFILL_TFLOPS_PER_SM = 3.75


def concurrent_decode_sms(decode_bytes: float, prefill_flops: float, sms: int) -> int:
    """SMs for the decode when it runs beside the chunk prefill on the others."""
    best = None
    for d in range(1, sms):
        t_dec = decode_bytes / (min(d * DECODE_GBS_PER_SM, DECODE_GBS_MAX) * 1e9)
        t_pre = prefill_flops / ((sms - d) * PREFILL_TFLOPS_PER_SM * 1e12)
        t = max(t_dec, t_pre)
        if best is None or t < best[0]:
            best = (t, d)
    return best[1]


def workload(key: str, layers=None, seed_offset=0):
    from paged_kv_cache_299_gb300 import workloads as wl
    make = wl.WORKLOADS[key]
    w = make() if not seed_offset else make(seed=make().seed + seed_offset)
    if layers is not None:
        w.layers = int(layers)
    return w


def describe(w) -> dict:
    ctx = w.context_lens
    d = {"workload": w.name, "batch": int(w.num_seqs), "layers": int(w.layers),
         "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
         "block_size": w.block_size, "prefill_chunks": int(w.num_prefill),
         "decode_seqs": int(w.num_decode), "context_min": int(ctx.min()),
         "context_max": int(ctx.max()), "context_mean": round(float(ctx.mean()), 1),
         "new_tokens_per_step": int(w.new_lens.sum()), "pool_blocks_per_layer": int(w.num_blocks),
         "kv_read_bytes_per_step": int(w.decode_kv_bytes()),
         "partition_tokens": int(w.partition_tokens)}
    return d


# ----------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling every 20 ms, started ahead of the region it measures (the tool
    needs a moment to start); mark() brackets the region, and stop() keeps the samples whose
    timestamps fall inside it."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    TIME_FORMAT = "%Y/%m/%d %H:%M:%S.%f"

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None
        self.t0 = None
        self.t1 = None

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.seek(0)
        return self.summarise(self.file.read(), self.t0, self.t1)

    @classmethod
    def summarise(cls, text: str, t0=None, t1=None) -> dict:
        """Median SM clock, maximum clock and the throttle reasons seen, over the samples
        between t0 and t1 (all samples when no bound is set or none falls inside)."""
        rows = []
        for line in text.strip().splitlines():
            r = [x.strip() for x in line.split(",")]
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], cls.TIME_FORMAT)
                rows.append((ts, float(r[2]), float(r[3]), r[6:10]))
            except ValueError:
                continue
        inside = [x for x in rows
                  if (t0 is None or x[0] >= t0) and (t1 is None or x[0] <= t1)]
        window = "the marked region"
        if not inside:
            inside, window = rows, "the whole sampling (no sample inside the marked region)"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {name for _, _, _, vals in inside
                   for name, val in zip(names, vals) if val.lower() == "active"}
        sm = [x[1] for x in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(x[2] for x in inside) if inside else None,
                "samples": len(sm), "reasons": sorted(reasons), "samples_from": window}


# ----------------------------------------------------------------------------------------
# the GB300 arm
# ----------------------------------------------------------------------------------------
def carve(torch, dev, specs):
    """Tensors (name, shape, dtype) carved out of one device buffer at 256-byte offsets, so
    that a step's inputs, or its outputs, cross the host link in a single copy."""
    views, offs, total = {}, [], 0
    for name, shape, dt in specs:
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        offs.append((name, shape, dt, total, nbytes))
        total += (nbytes + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    for name, shape, dt, o, n in offs:
        views[name] = buf[o:o + n].view(dt).view(shape)
    return buf, views


class DeviceStep:
    """Resident state of one workload: per-layer pools (history already stored through the
    library), workspaces, and one or more sets of this step's input and output buffers."""

    def __init__(self, w, dev, fused_append=False, mixed="split"):
        import torch
        from paged_kv_cache_299_gb300 import binding as pa
        self.pa = pa
        self.torch = torch
        self.w = w
        self.dev = dev
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
        self.n_pre_rows = int(w.prefill_query_start_loc[-1]) if w.num_prefill else 0
        self.n_rows = self.n_pre_rows + w.num_decode
        self.n_new = int(w.new_lens.sum())
        # every per-step input (queries, new K/V of each layer, block tables, context
        # lengths) lives in one device buffer, every output in another
        bf = torch.bfloat16
        self.in_specs = []
        for layer in range(w.layers):
            self.in_specs += [(f"q{layer}", (self.n_rows, w.num_q_heads, w.head_dim), bf),
                              (f"k{layer}", (self.n_new, w.num_kv_heads, w.head_dim), bf),
                              (f"v{layer}", (self.n_new, w.num_kv_heads, w.head_dim), bf)]
        self.in_specs += [("bt", tuple(w.block_tables.shape), torch.int32),
                          ("ctx", (w.num_seqs,), torch.int32)]
        self.out_specs = [(f"o{layer}", (self.n_rows, w.num_q_heads, w.head_dim), bf)
                          for layer in range(w.layers)]
        self.sets = [self._carve_set()]
        S = self.sets[0]
        S["bt"].copy_(i32(w.block_tables))
        S["ctx"].copy_(i32(w.context_lens))
        self.new_qsl = i32(w.new_start_loc)
        self.one_token_each = bool((w.new_lens == 1).all())
        # one new token per decode sequence and no prefill: the store can ride in the decode
        self.fused_append = bool(fused_append and self.one_token_each and w.num_prefill == 0)
        self.pre_qsl = i32(w.prefill_query_start_loc)
        self.max_ctx_dec = int(w.decode_context_lens.max()) if w.num_decode else 0
        self.max_q_pre = int(w.new_lens[: w.num_prefill].max()) if w.num_prefill else 0
        # unified: one varlen call serves the chunks (first) and the decode rows of a step
        self.unified = bool(mixed == "unified" and w.num_prefill and w.num_decode
                            and self.one_token_each is False)
        # concurrent: the decode on decode_sms SMs, the chunk prefill beside it on the rest
        self.concurrent = bool(mixed == "concurrent" and w.num_prefill and w.num_decode)
        self.all_qsl = i32(np.concatenate([w.prefill_query_start_loc[: w.num_prefill + 1]
                                           if w.num_prefill else [0],
                                           self.n_pre_rows + np.arange(1, w.num_decode + 1)]))
        self.status = pa.new_device_status(dev)
        self.slots = torch.empty(self.n_new, dtype=torch.int64, device=dev)
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        self.pools = []
        hist_ctx = i32(w.hist_lens)
        hist_qsl = i32(w.hist_start_loc)
        n_hist = int(w.hist_lens.sum())
        for layer in range(w.layers):
            vals = w.values(layer, dev)
            kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev)
            vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev)
            if n_hist:
                hs = pa.pa_compute_slot_mapping(S["bt"], hist_ctx, hist_qsl, n_hist, kc,
                                                device_status=self.status)
                pa.pa_reshape_and_cache(vals["hist_k"], vals["hist_v"], hs, kc, vc,
                                        device_status=self.status)
                del hs
            self.pools.append((kc, vc))
            L = S["layers"][layer]
            L["q_all"].copy_(torch.cat([vals["q_prefill"], vals["q_decode"]]))
            L["new_k"].copy_(vals["new_k"])
            L["new_v"].copy_(vals["new_v"])
            del vals
            torch.cuda.synchronize(dev)
        # the library merges split-KV pieces inside the decode kernel up to 8192-token
        # contexts with automatic partitions; otherwise a second (merge) kernel runs
        self.ws_merge_kernel = bool(w.partition_tokens > 0 or self.max_ctx_dec > 8192)
        if self.unified:
            self.ws_var = torch.empty(pa.pa_varlen_workspace_size(w.num_seqs, self.n_rows),
                                      dtype=torch.uint8, device=dev)
        if w.num_decode:
            need = pa.pa_decode_workspace_size(w.num_decode, w.num_kv_heads, w.num_q_heads,
                                               self.max_ctx_dec, w.partition_tokens)
            self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
        if self.concurrent or self.unified:
            # (the unified call takes the same split: decode rows on decode_sms SMs)
            self.sms = torch.cuda.get_device_properties(dev).multi_processor_count
            self.decode_sms = concurrent_decode_sms(w.decode_kv_bytes() / w.layers,
                                                    self.prefill_flops() / w.layers, self.sms)
        assert pa.pa_check_device_status(self.status) == pa.PA_OK

    def _carve_set(self) -> dict:
        """One set of step buffers: queries / new K/V / tables in one device buffer, outputs
        in another; queries and outputs of all rows per layer, chunks first, the per-kind
        tensors being views."""
        torch, dev, w, npre = self.torch, self.dev, self.w, self.n_pre_rows
        inbuf, inv = carve(torch, dev, self.in_specs)
        outbuf, outv = carve(torch, dev, self.out_specs)
        S = {"inbuf": inbuf, "outbuf": outbuf, "bt": inv["bt"], "ctx": inv["ctx"], "layers": []}
        S["bt_dec"], S["ctx_dec"] = S["bt"][w.num_prefill:], S["ctx"][w.num_prefill:]
        S["bt_pre"], S["ctx_pre"] = S["bt"][: w.num_prefill], S["ctx"][: w.num_prefill]
        for layer in range(w.layers):
            q_all, out_all = inv[f"q{layer}"], outv[f"o{layer}"]
            S["layers"].append({
                "new_k": inv[f"k{layer}"], "new_v": inv[f"v{layer}"],
                "q_all": q_all, "out_all": out_all,
                "q_pre": q_all[:npre], "q_dec": q_all[npre:],
                "out_pre": out_all[:npre], "out_dec": out_all[npre:],
            })
        return S

    def add_buffer_set(self) -> int:
        """A second set of step buffers holding the same inputs (for overlapped copies)."""
        S = self._carve_set()
        S["inbuf"].copy_(self.sets[0]["inbuf"])
        self.sets.append(S)
        return len(self.sets) - 1

    def launches_per_step(self) -> int:
        w = self.w
        if self.fused_append:
            return w.layers * (2 if self.ws_merge_kernel else 1)
        if self.unified:  # store; per layer the decode rows' kernel (+ merge) and the chunk kernel
            return 1 + (3 if self.ws_merge_kernel else 2) * w.layers
        per_layer = 1 + ((2 if self.ws_merge_kernel else 1) if w.num_decode else 0) + \
            (1 if w.num_prefill else 0)
        return 1 + per_layer * w.layers

    def prefill_flops(self) -> float:
        """Causal-useful flops of this step's prefill chunks: row i of a chunk over h prior
        tokens attends h + i + 1 keys; 4 * head_dim flops per (row, head, key)."""
        w = self.w
        h = w.hist_lens[: w.num_prefill].astype(np.float64)
        n = w.new_lens[: w.num_prefill].astype(np.float64)
        keys = (n * h + n * (n + 1) / 2).sum()
        return float(keys * w.num_q_heads * 4 * w.head_dim * w.layers)

    def step(self, dec_events=None, pre_events=None, set_idx=0):
        pa, w = self.pa, self.w
        S = self.sets[set_idx]
        if self.fused_append:
            for li, L in enumerate(S["layers"]):
                kc, vc = self.pools[li]
                if dec_events is not None:
                    dec_events[li][0].record()
                # each layer after the first follows the previous layer's decode, which
                # writes other pools: its start-up may overlap that kernel's last CTAs
                flags = pa.PA_LAUNCH_OVERLAP_PREVIOUS if li > 0 else pa.PA_LAUNCH_DEFAULT
                pa.pa_decode_append(L["out_dec"], L["q_dec"], L["new_k"], L["new_v"], kc, vc,
                                    S["bt_dec"], S["ctx_dec"], w.scale, self.max_ctx_dec,
                                    w.partition_tokens, workspace=self.ws, launch_flags=flags)
                if dec_events is not None:
                    dec_events[li][1].record()
            return
        pa.pa_compute_slot_mapping(S["bt"], S["ctx"],
                                   None if self.one_token_each else self.new_qsl, self.n_new,
                                   self.pools[0][0], slot_mapping=self.slots)
        for li, L in enumerate(S["layers"]):
            kc, vc = self.pools[li]
            pa.pa_reshape_and_cache(L["new_k"], L["new_v"], self.slots, kc, vc)
            if self.unified:
                if dec_events is not None:
                    dec_events[li][0].record()
                pa.pa_attention_varlen(L["out_all"], L["q_all"], self.all_qsl,
                                       max(self.max_q_pre, 1), kc, vc, S["bt"], S["ctx"],
                                       w.scale, workspace=self.ws_var,
                                       launch_flags=pa.PA_LAUNCH_MAX_SMS(self.decode_sms))
                if dec_events is not None:
                    dec_events[li][1].record()
                continue
            if self.concurrent:
                # the decode on decode_sms SMs, then the chunk prefill starting at once on
                # the other SMs (it writes and reads nothing the decode touches)
                pa.pa_decode(L["out_dec"], L["q_dec"], kc, vc, S["bt_dec"], S["ctx_dec"],
                             w.scale, self.max_ctx_dec, w.partition_tokens, workspace=self.ws,
                             launch_flags=pa.PA_LAUNCH_MAX_SMS(self.decode_sms))
                pa.pa_prefill_chunk(L["out_pre"], L["q_pre"], self.pre_qsl, self.max_q_pre,
                                    kc, vc, S["bt_pre"], S["ctx_pre"], w.scale,
                                    launch_flags=pa.PA_LAUNCH_OVERLAP_PREVIOUS |
                                    pa.PA_LAUNCH_MAX_SMS(self.sms - self.decode_sms))
                continue
            if w.num_prefill:
                if pre_events is not None:
                    pre_events[li][0].record()
                pa.pa_prefill_chunk(L["out_pre"], L["q_pre"], self.pre_qsl, self.max_q_pre,
                                    kc, vc, S["bt_pre"], S["ctx_pre"], w.scale)
                if pre_events is not None:
                    pre_events[li][1].record()
            if w.num_decode:
                if dec_events is not None:
                    dec_events[li][0].record()
                # after the chunk prefill, which writes only its own output rows, the
                # decode's start-up may overlap the prefill's last CTAs
                flags = pa.PA_LAUNCH_OVERLAP_PREVIOUS if w.num_prefill else pa.PA_LAUNCH_DEFAULT
                pa.pa_decode(L["out_dec"], L["q_dec"], kc, vc, S["bt_dec"], S["ctx_dec"],
                             w.scale, self.max_ctx_dec, w.partition_tokens, workspace=self.ws,
                             launch_flags=flags)
                if dec_events is not None:
                    dec_events[li][1].record()


def make_flush(dev, kv_bytes: int, mode: str):
    """L2 flush between steps for workloads smaller than 4x L2 (None for larger ones):
    rewrite a buffer of twice the L2 size, then (write-read) read another one, so that the
    dirty lines are written back before the step rather than during it."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    if kv_bytes >= 4 * l2:
        return None
    buf = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)
    rd = torch.zeros(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev) \
        if mode == "write-read" else None

    def flush_l2(k):
        buf.fill_(k)
        if rd is not None:
            rd.sum()
    return flush_l2


def time_steps(st, dev, K: int, warmup: int, flush_l2, use_graph: bool, barrier=None,
               sampler=None) -> dict:
    """W untimed steps, then K timed steps (one CUDA-graph replay or eager C-ABI calls each,
    events on the launching stream, L2 flushed before each when flush_l2 is given); then
    per-kernel event times from an eager pass of min(K, 20) steps of the same workload."""
    import torch
    w = st.w
    barrier = barrier or (lambda: None)
    for _ in range(warmup):
        st.step()
    torch.cuda.synchronize(dev)
    barrier()
    n_kernel = min(K, 20) if use_graph else K
    mk = lambda: [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    # (a concurrent step's kernels overlap: no per-kernel events)
    dec_ev = [[mk() for _ in range(w.layers)] for _ in range(K)] \
        if w.num_decode and not st.concurrent else None
    pre_ev = [[mk() for _ in range(w.layers)] for _ in range(K)] \
        if w.num_prefill and not st.unified and not st.concurrent else None
    step_ev = [mk() for _ in range(K)]
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)
    torch.cuda.synchronize(dev)
    barrier()
    graph = None
    if use_graph:
        from paged_kv_cache_299_gb300 import graphs
        graph = graphs.StepGraph(st.step)
    if sampler is not None:
        sampler.mark_start()
    t_wall = time.perf_counter()
    for k in range(K):
        if flush_l2 is not None:
            flush_l2(k)
        step_ev[k][0].record()
        if graph is not None:
            graph.replay()
        else:
            st.step(dec_ev[k] if dec_ev else None, pre_ev[k] if pre_ev else None)
        step_ev[k][1].record()
    torch.cuda.synchronize(dev)
    if graph is not None and dec_ev:  # per-kernel timing: an eager pass right after
        for k in range(n_kernel):
            if flush_l2 is not None:
                flush_l2(k)
            st.step(dec_ev[k] if dec_ev else None, pre_ev[k] if pre_ev else None)
        torch.cuda.synchronize(dev)
    barrier()
    wall = time.perf_counter() - t_wall
    res = {"step_ms": sum(a.elapsed_time(b) for a, b in step_ev) / K, "wall": wall,
           "graph": graph, "clocks": None, "dec_ms": None, "pre_ms": None}
    if dec_ev:
        res["dec_ms"] = sum(a.elapsed_time(b) for row in dec_ev[:n_kernel] for a, b in row) / (
            n_kernel * w.layers)
    if pre_ev:
        res["pre_ms"] = sum(a.elapsed_time(b) for row in pre_ev[:n_kernel] for a, b in row) / (
            n_kernel * w.layers)
    return res


def decode_roofline(st, workload_key: str, dec_ms: float, peak: float, peak_src: str,
                    step_ms: float | None = None) -> dict:
    """Roofline of the decode kernel.  When the timed step is nothing but one fused decode
    launch per layer (several layers), the launch duration is the timed region's time per
    launch: there consecutive layers overlap (PA_LAUNCH_OVERLAP_PREVIOUS), so one launch
    between two events of its own would not show what the step sustains.  That isolated
    figure (an eager pass right after the timed region) is reported beside it."""
    w = st.w
    if getattr(st, "concurrent", False):
        # the decode and the chunk prefill overlap: the step's time per layer bounds the
        # decode's own duration from above (a conservative figure)
        per_launch = w.decode_kv_bytes() / w.layers
        launch_ms = step_ms / w.layers
        achieved = per_launch / (launch_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic("paged_decode_kernel", workload_key),
                "kernel": f"pa_decode on {st.decode_sms} SMs beside the chunk prefill",
                "peak_source": f"{peak_src} hbm_gbs", "launch_ms": round(launch_ms, 5),
                "algorithmic_bytes_per_launch": int(per_launch),
                "timing": "timed region / layers: the decode runs beside the chunk prefill, "
                          "so the step's time per layer stands for its duration"}
    if st.unified:
        # the varlen launch reads the K/V of every sequence of the step at least once
        per_launch = float(np.sum(w.context_lens)) * w.num_kv_heads * w.head_dim * 2 * 2
        achieved = per_launch / (dec_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": None,
                "kernel": "pa_attention_varlen: paged_decode_kernel over the decode rows, "
                          "paged_prefill_kernel (tcgen05) over the chunks",
                "peak_source": f"{peak_src} hbm_gbs", "launch_ms": round(dec_ms, 5),
                "algorithmic_bytes_per_launch": int(per_launch)}
    per_launch = w.decode_kv_bytes() / w.layers
    isolated = per_launch / (dec_ms * 1e-3) / 1e9
    region = (step_ms is not None and st.fused_append and w.layers > 1 and not w.num_prefill
              and not st.ws_merge_kernel)
    launch_ms = step_ms / w.layers if region else dec_ms
    achieved = per_launch / (launch_ms * 1e-3) / 1e9
    out = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
           "frac": round(achieved / peak, 4),
           "traffic": ncu_traffic("paged_decode_kernel", workload_key),
           "kernel": "pa_decode: paged_decode_kernel (split-KV merge in-kernel up to "
                     "8192-token contexts, else + merge_partials_kernel)",
           "peak_source": f"{peak_src} hbm_gbs", "pct_of_8tbs": round(100 * achieved / 8000, 2),
           "launch_ms": round(launch_ms, 5), "algorithmic_bytes_per_launch": int(per_launch),
           "timing": ("timed region / decode launches in it (the step is only these "
                      "launches, consecutive layers overlapping)" if region else
                      "eager pass right after the timed region, each launch between two "
                      "events")}
    if region:
        out["isolated"] = {"achieved": round(isolated, 1), "frac": round(isolated / peak, 4),
                           "launch_ms": round(dec_ms, 5),
                           "timing": "eager pass right after the timed region, each launch "
                                     "between two events"}
    return out


def prefill_roofline(st, pre_ms: float) -> dict:
    w = st.w
    tfl = st.prefill_flops() / w.layers / (pre_ms * 1e-3) / 1e12
    bf16_peak, bf16_src = measured_bf16_peak()
    return {"bound": "tensor", "achieved": round(tfl, 1), "peak": bf16_peak, "unit": "TFLOP/s",
            "frac": round(tfl / bf16_peak, 4), "kernel": "paged_prefill_kernel (tcgen05)",
            "peak_source": f"{bf16_src} bf16_tflops_sustained", "launch_ms": round(pre_ms, 5),
            "algorithmic_flops_per_launch": round(st.prefill_flops() / w.layers)}


def run_gpu(args, rank, world):
    import torch
    import torch.distributed as dist

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # weak scaling: every rank serves its own batch (seed offset per rank)
    w = workload(args.workload, args.layers, 100 * rank if world > 1 else 0)
    st = DeviceStep(w, dev, fused_append=args.append == "fused", mixed=args.mixed)
    kv_bytes = w.decode_kv_bytes()
    flush_l2 = make_flush(dev, kv_bytes, args.flush)

    def barrier():
        if world > 1:
            dist.barrier()

    K = args.steps
    # clocks are sampled from just before the timed steps to the end of the end-to-end
    # loop, so that short timed regions still get several samples under load
    sampler = ClockSampler(local)
    t = time_steps(st, dev, K, args.warmup, flush_l2, args.launch == "graph", barrier, sampler)
    graph = t["graph"]
    # the in-run read reference: one launch reading as many bytes as one decode launch,
    # under the same L2 rule, timed the same way
    stream_ref = None
    if w.num_decode and not st.unified:
        stream_ref = measure_stream_read(dev, kv_bytes // w.layers, flush_l2, max(3, min(K, 20)))
    step_ms = max_over_ranks(t["step_ms"], dev)

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(st, max(3, min(K, 50)), dev, graph, flush_l2)
        e2e["step_ms"] = max_over_ranks(e2e["step_ms"], dev)
    torch.cuda.synchronize(dev)
    sampler.mark_end()
    t["clocks"] = dict(sampler.stop(), window="from the timed steps to the end of the "
                                              "end-to-end loop")

    if rank != 0:
        return
    peak, peak_src = measured_peaks()
    value = whole_job_gbs(kv_bytes, world, step_ms)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": dict(describe(w), parallelism=f"replicas{world}" if world > 1 else "single",
                       accumulate="f32",
                       l2=(("flushed between steps (2x L2 rewrite, then 2x L2 read)"
                            if args.flush == "write-read" else
                            "flushed between steps (2x L2 rewrite)") if flush_l2
                           else "inputs larger than L2 (%.1f GB KV per step)" % (kv_bytes / 1e9)),
                       launch=("CUDA graph: one replay per step (kernel times from an "
                               "eager pass right after)" if graph is not None
                               else "eager (one C-ABI call per kernel group)"),
                       store=("fused into decode (pa_decode_append)" if st.fused_append
                              else "pa_compute_slot_mapping + pa_reshape_and_cache"),
                       **({"overlap": "layers after the first start under programmatic "
                                      "dependent launch (PA_LAUNCH_OVERLAP_PREVIOUS)"}
                          if st.fused_append and w.layers > 1 else
                          {"overlap": f"the decode on {st.decode_sms} SMs "
                                      "(PA_LAUNCH_MAX_SMS), the chunk prefill beside it on "
                                      f"the other {st.sms - st.decode_sms} "
                                      "(PA_LAUNCH_OVERLAP_PREVIOUS)"}
                          if st.concurrent else
                          {"overlap": f"one varlen call: decode rows on {st.decode_sms} SMs, "
                                      f"the chunks beside them on the other "
                                      f"{st.sms - st.decode_sms}"}
                          if st.unified else
                          {"overlap": "the decode starts under programmatic dependent launch "
                                      "behind the chunk prefill (PA_LAUNCH_OVERLAP_PREVIOUS)"}
                          if w.num_prefill and w.num_decode and not st.unified else {}),
                       **({"attention": "pa_attention_varlen: decode rows on the decode "
                                        "kernel, chunks on the tensor-core kernel"}
                          if st.unified else {})),
        "tokens_per_s": round(w.num_decode * world / (step_ms * 1e-3), 1),
        "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "gpu_launches": st.launches_per_step() * K,
        "wall_s_timed": round(t["wall"], 3),
        "clocks": t["clocks"],
    }
    if t["dec_ms"] or st.concurrent:
        res["roofline"] = decode_roofline(st, args.workload, t["dec_ms"], peak, peak_src,
                                          step_ms=t["step_ms"])
    if stream_ref and "roofline" in res:
        res["roofline"]["stream_read"] = dict(
            stream_ref, decode_frac_of_stream=round(res["roofline"]["achieved"] /
                                                    stream_ref["achieved"], 4))
    if t["pre_ms"]:
        res["prefill_roofline"] = prefill_roofline(st, t["pre_ms"])
    if e2e:
        res["e2e"] = {"value": round(whole_job_gbs(kv_bytes, world, e2e["step_ms"]), 1),
                      "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"],
                      "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": round(e2e["step_ms"], 4)}
    del st, graph, t
    torch.cuda.empty_cache()
    if not args.no_secondary and world == 1:
        res["secondary"] = run_secondary(args, dev, local, peak, peak_src)
    if not args.no_cpu_baseline and world == 1:
        res["cpu_baseline"] = cpu_baseline(w, target_s=10.0)
        res["cpu_baseline_all_cores"] = cpu_baseline_all_cores(w, target_s=10.0)
    print(json.dumps(res), flush=True)


# The other workloads, measured in the same invocation with the same method (graph-replayed
# step, eager per-kernel events, in-run stream read of one decode launch's bytes), and a
# standalone KV store: (name, workload, timed steps, layers or None for the workload's own).
# The batch-64 decode is measured twice: one layer with L2 flushed before every step (one
# launch alone), and back to back over 16 layers, each with its own pool (2.2 GB per step,
# no flush), the later layers overlapping the earlier ones as in the default step.  The
# mixed step is measured twice too: chunk prefill then decode (each kernel on every SM,
# timed one by one), and the decode on part of the SMs with the chunk prefill beside it.
SECONDARY = (("single_seq_300", "single_seq_300", 200, None, "split"),
             ("decode_b64", "decode_b64", 100, None, "split"),
             ("decode_b64_16layers", "decode_b64", 50, 16, "split"),
             ("long_context_b4", "long_context_b4", 30, None, "split"),
             ("mixed_step", "mixed_step", 30, None, "split"),
             ("mixed_step_concurrent", "mixed_step", 30, None, "concurrent"))


def run_secondary(args, dev, local: int, peak: float, peak_src: str) -> dict:
    import torch
    out = {}
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    sampler.mark_start()
    for name, key, K, layers, mixed in SECONDARY:
        if key == args.workload and layers is None and mixed == args.mixed:
            continue
        w = workload(key, layers)
        st = DeviceStep(w, dev, fused_append=True, mixed=mixed)
        kv = w.decode_kv_bytes()
        flush_l2 = make_flush(dev, kv, "write-read")
        t = time_steps(st, dev, K, 3, flush_l2, True)
        d = {"kv_read_bytes_per_step": kv, "steps": K, "ms_per_step": round(t["step_ms"], 5),
             "us_per_step": round(t["step_ms"] * 1e3, 2),
             "step_gbs": round(kv / (t["step_ms"] * 1e-3) / 1e9, 1),
             "step_pct_of_8tbs": round(100 * kv / (t["step_ms"] * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 2),
             "l2": "flushed between steps" if flush_l2 else "inputs larger than L2",
             "store": ("fused into decode (pa_decode_append)" if st.fused_append
                       else "pa_compute_slot_mapping + pa_reshape_and_cache")}
        if layers is not None:
            d["layers"] = int(w.layers)
        if st.concurrent:
            d["schedule"] = (f"decode on {st.decode_sms} SMs (PA_LAUNCH_MAX_SMS), chunk prefill "
                             f"beside it on the other {st.sms - st.decode_sms} "
                             "(PA_LAUNCH_OVERLAP_PREVIOUS); the kernels overlap, so no "
                             "per-kernel times")
            d["prefill_tflops_over_step"] = round(
                st.prefill_flops() / (t["step_ms"] * 1e-3) / 1e12, 1)
        if t["dec_ms"]:
            d["roofline"] = decode_roofline(st, key, t["dec_ms"], peak, peak_src,
                                            step_ms=t["step_ms"])
            # one launch's bytes, flushed before each read when they fit in 4x L2
            sr = measure_stream_read(dev, kv // w.layers,
                                     make_flush(dev, kv // w.layers, "write-read"), 20)
            d["roofline"]["stream_read"] = dict(
                sr, decode_frac_of_stream=round(d["roofline"]["achieved"] / sr["achieved"], 4))
        if t["pre_ms"]:
            d["prefill_roofline"] = prefill_roofline(st, t["pre_ms"])
        out[name] = d
        del st, t
        torch.cuda.empty_cache()
    out["reshape_and_cache"] = measure_store(dev, peak, peak_src)
    out["copy_blocks"] = measure_copy_blocks(dev, peak, peak_src)
    sampler.mark_end()
    out["clocks"] = sampler.stop()
    return out


def _event_ms(dev, fn, reps: int, flush_l2=None) -> float:
    """Mean CUDA-event time of fn() over reps launches (3 untimed first)."""
    import torch
    for _ in range(3):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i, (a, b) in enumerate(evs):
        if flush_l2 is not None:
            flush_l2(i)
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in evs) / reps


def measure_copy_blocks(dev, peak: float, peak_src: str, pairs: int = 8192) -> dict:
    """pa_copy_blocks alone: `pairs` copy-on-write block copies (source and destination
    blocks drawn without replacement from a shuffled pool of 2 x pairs + 10 % blocks).
    Algorithmic bytes per pair: the K and V blocks (8 heads x 16 x 64 bf16 = 16 KiB each)
    read and written, 64 KiB."""
    import torch
    from paged_kv_cache_299_gb300 import binding as pa
    nb = int(2 * pairs * 1.1)
    perm = np.random.default_rng(88).permutation(nb)[: 2 * pairs].astype(np.int64)
    mapping = torch.from_numpy(perm.reshape(pairs, 2)).to(dev)
    shape = (nb, 8, 16, 64)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    nbytes = pairs * 4 * 8 * 16 * 64 * 2
    flush_l2 = make_flush(dev, nbytes, "write-read")
    ms = _event_ms(dev, lambda: pa.pa_copy_blocks(kc, vc, mapping), 50, flush_l2)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del kc, vc
    torch.cuda.empty_cache()
    return {"pairs": pairs, "algorithmic_bytes_per_launch": nbytes, "launch_ms": round(ms, 5),
            "achieved": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / peak, 4),
            "peak_source": f"{peak_src} hbm_gbs", "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
            "traffic": ncu_traffic("copy_blocks_kernel", f"pairs_{pairs}"),
            "l2": "flushed before each launch" if flush_l2 else "inputs larger than L2"}


def measure_store(dev, peak: float, peak_src: str) -> dict:
    """pa_reshape_and_cache alone, CUDA events per launch: the mixed step's 4344 new tokens
    (the largest per-step store of the workloads; L2 flushed before each launch) and a bulk
    store of 65536 tokens (8 prompts of 8192, e.g. a large prefill).  Algorithmic bytes per
    token: 2 x 1024 B read (K and V rows of 8 heads) + 2 x 1024 B written."""
    import torch
    from paged_kv_cache_299_gb300 import binding as pa
    from paged_kv_cache_299_gb300 import workloads as wl
    res = {}
    cases = (("mixed_step_4344_tokens", wl.mixed_prefill_decode()),
             ("bulk_65536_tokens", wl.make_workload("bulk_store", [0] * 8, [8192] * 8,
                                                    num_prefill=8, seed=77)))
    for name, w in cases:
        vals = w.values(0, dev)
        k, v = vals["new_k"], vals["new_v"]
        del vals
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        vc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        bt = torch.from_numpy(w.block_tables).to(dev)
        ctx = torch.from_numpy(w.context_lens).to(dev)
        qsl = torch.from_numpy(w.new_start_loc).to(dev)
        n = int(w.new_lens.sum())
        slots = pa.pa_compute_slot_mapping(bt, ctx, qsl, n, kc)
        nbytes = n * w.num_kv_heads * w.head_dim * 2 * 2 * 2
        flush_l2 = make_flush(dev, nbytes, "write-read")
        ms = _event_ms(dev, lambda: pa.pa_reshape_and_cache(k, v, slots, kc, vc), 50, flush_l2)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"tokens": n, "algorithmic_bytes_per_launch": nbytes,
                     "launch_ms": round(ms, 5), "achieved": round(gbs, 1), "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_source": f"{peak_src} hbm_gbs",
                     "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
                     "traffic": ncu_traffic("reshape_and_cache_kernel", name),
                     "l2": "flushed before each launch" if flush_l2 else "inputs larger than L2"}
        del k, v, kc, vc, slots
        torch.cuda.empty_cache()
    return res


def measure_stream_read(dev, nbytes: int, flush_l2, reps: int) -> dict:
    """pa_stream_read over `nbytes` (one decode launch's KV bytes): 16-byte vector loads of a
    contiguous buffer in one launch, CUDA events around each launch (L2 flushed before each
    when the decode's workload is flushed)."""
    import torch
    from paged_kv_cache_299_gb300 import binding as pa

    nbytes -= nbytes % 16
    buf = torch.zeros(nbytes // 4, dtype=torch.int32, device=dev)
    x = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        pa.pa_stream_read(buf, x)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for k, (a, b) in enumerate(evs):
        if flush_l2 is not None:
            flush_l2(k)
        a.record()
        pa.pa_stream_read(buf, x)
        b.record()
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in evs) / reps
    del buf
    return {"achieved": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "bytes": nbytes,
            "launch_ms": round(ms, 5),
            "kernel": "pa_stream_read: one launch of 16-byte streaming loads over a contiguous "
                      "buffer of one decode launch's KV bytes"}


def run_e2e(st: DeviceStep, steps: int, dev, graph=None, flush_l2=None) -> dict:
    """Each step: pinned host -> device copy of the step's inputs (queries, new K/V, block
    tables, context lengths of every layer: one buffer), the step through the C ABI, and
    a device -> host copy of its attention outputs (one buffer).  As a serving loop would,
    two buffer sets alternate so that the copies of one step overlap the attention of its
    neighbour: inputs of step k+1 go up and outputs of step k-1 come down on two copy
    streams while step k computes.  Timed on the device from the first upload to the last
    download.  For workloads that must have L2 flushed between steps (flush_l2 given) the
    steps run one after the other instead, each timed from its upload to its download with
    the flush outside."""
    import torch
    n_sets = 2
    while len(st.sets) < n_sets:
        st.add_buffer_set()
    graphs = [graph] + [None] * (n_sets - 1)
    if graph is not None:
        from paged_kv_cache_299_gb300 import graphs as gmod
        for i in range(1, n_sets):
            graphs[i] = gmod.StepGraph(lambda i=i: st.step(set_idx=i))
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
    host_in = [pin(S["inbuf"]) for S in st.sets[:n_sets]]
    host_out = [torch.empty(S["outbuf"].shape, dtype=S["outbuf"].dtype, pin_memory=True)
                for S in st.sets[:n_sets]]
    h2d = host_in[0].numel() * host_in[0].element_size()
    d2h = host_out[0].numel() * host_out[0].element_size()
    compute = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(n_sets)]
    ev_done = [torch.cuda.Event() for _ in range(n_sets)]
    ev_out = [torch.cuda.Event() for _ in range(n_sets)]

    def run(k0, k1):
        for k in range(k0, k1):
            i = k % n_sets
            S = st.sets[i]
            with torch.cuda.stream(up):
                if k >= n_sets:  # step k - n_sets has finished with this set and its download
                    up.wait_event(ev_out[i])
                S["inbuf"].copy_(host_in[i], non_blocking=True)
                ev_in[i].record(up)
            compute.wait_event(ev_in[i])
            if graphs[i] is not None:
                graphs[i].replay()
            else:
                st.step(set_idx=i)
            ev_done[i].record(compute)
            with torch.cuda.stream(down):
                down.wait_event(ev_done[i])
                host_out[i].copy_(S["outbuf"], non_blocking=True)
                ev_out[i].record(down)
        compute.wait_stream(down)

    if flush_l2 is not None:
        S = st.sets[0]
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for k in range(2 + steps):
            flush_l2(k)
            if k >= 2:
                evs[k - 2][0].record(compute)
            S["inbuf"].copy_(host_in[0], non_blocking=True)
            if graphs[0] is not None:
                graphs[0].replay()
            else:
                st.step(set_idx=0)
            host_out[0].copy_(S["outbuf"], non_blocking=True)
            if k >= 2:
                evs[k - 2][1].record(compute)
        torch.cuda.synchronize(dev)
        return {"step_ms": sum(a.elapsed_time(b) for a, b in evs) / steps, "h2d": h2d,
                "d2h": d2h}
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    run(0, 2)
    torch.cuda.synchronize(dev)
    up.wait_stream(compute)
    start.record(compute)
    up.wait_event(start)
    run(0, steps)
    end.record(compute)
    torch.cuda.synchronize(dev)
    return {"step_ms": start.elapsed_time(end) / steps, "h2d": h2d, "d2h": d2h}


# ----------------------------------------------------------------------------------------
# the CPU oracle (baseline leg and --impl reference)
# ----------------------------------------------------------------------------------------
def oracle_sample(w, max_seqs: int, threads: int = 1):
    """A bounded sample of the workload: its first sequences (same length law), one layer,
    drawn on the host; returns a callable doing one oracle step and its KV bytes.  With
    threads > 1 the step's attention runs on that many host threads, each over a disjoint
    slice of the sequences (the oracle itself is unchanged: ctypes releases the GIL during
    each call and the oracle keeps no shared state)."""
    import concurrent.futures as cf

    import oracle
    from paged_kv_cache_299_gb300 import workloads as wl

    n = min(max_seqs, w.num_seqs)
    npre = min(w.num_prefill, n)
    sw = wl.make_workload(w.name + f"_sample{n}", w.hist_lens[:n], w.new_lens[:n],
                          num_prefill=npre, seed=w.seed,
                          big_key_fraction=w.big_key_fraction)
    vals = sw.values(0, "cpu")
    kc, vc = wl.nan_pool(sw.num_blocks), wl.nan_pool(sw.num_blocks)
    hs, err = oracle.slot_mapping(sw.block_tables, sw.hist_lens, sw.hist_start_loc, sw.num_blocks)
    oracle.reshape_and_cache(wl.bf16_bits(vals["hist_k"]), wl.bf16_bits(vals["hist_v"]), hs,
                             kc, vc)
    new_k, new_v = wl.bf16_bits(vals["new_k"]), wl.bf16_bits(vals["new_v"])
    qd, qp = wl.bf16_bits(vals["q_decode"]), wl.bf16_bits(vals["q_prefill"])
    dbt, dctx = sw.decode_block_tables, sw.decode_context_lens
    qsl = sw.prefill_query_start_loc
    pool = cf.ThreadPoolExecutor(max_workers=threads) if threads > 1 else None
    # units of work: one per prefill sequence, and decode slices of about equal size
    nd = sw.num_decode
    per = max(1, -(-nd // (4 * threads))) if nd else 1

    def prefill_one(s):
        oracle.prefill_chunk(qp[qsl[s]:qsl[s + 1]], np.array([0, qsl[s + 1] - qsl[s]], np.int32),
                             kc, vc, sw.block_tables[s:s + 1], sw.context_lens[s:s + 1], sw.scale)

    def decode_slice(a):
        b = min(nd, a + per)
        oracle.decode(qd[a:b], kc, vc, dbt[a:b], dctx[a:b], sw.scale)

    def step():
        slots, _ = oracle.slot_mapping(sw.block_tables, sw.context_lens, sw.new_start_loc,
                                       sw.num_blocks)
        oracle.reshape_and_cache(new_k, new_v, slots, kc, vc)
        if pool is None:
            if sw.num_prefill:
                oracle.prefill_chunk(qp, qsl, kc, vc, sw.block_tables[:npre],
                                     sw.context_lens[:npre], sw.scale)
            if nd:
                oracle.decode(qd, kc, vc, dbt, dctx, sw.scale)
            return
        futs = [pool.submit(prefill_one, s) for s in range(sw.num_prefill)]
        futs += [pool.submit(decode_slice, a) for a in range(0, nd, per)]
        for f in futs:
            f.result()

    return sw, step, sw.decode_kv_bytes()


def _timed_oracle(w, max_seqs: int, threads: int, target_s: float):
    sw, step, kv = oracle_sample(w, max_seqs, threads)
    step()  # warm
    reps, t0 = 0, time.perf_counter()
    while True:
        step()
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return sw, kv, reps, el


def cpu_baseline(w, target_s: float) -> dict:
    """The oracle as written: one host thread."""
    sw, kv, reps, el = _timed_oracle(w, 32, 1, target_s)
    return {"value": round(kv * reps / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"one layer of the first {sw.num_seqs} sequences of {w.name} "
                      f"({int(sw.context_lens.sum())} cached tokens), {reps} repetitions, "
                      f"{el:.1f} s single-threaded",
            "tokens_per_s": round(sw.num_decode * reps / el, 3)}


def cpu_baseline_all_cores(w, target_s: float) -> dict:
    """The same oracle on every host core: the step's sequences split over os.cpu_count()
    threads (disjoint slices, no shared state)."""
    cores = os.cpu_count() or 1
    sw, kv, reps, el = _timed_oracle(w, 256, cores, target_s)
    return {"value": round(kv * reps / el / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"one layer of the first {sw.num_seqs} sequences of {w.name} "
                      f"({int(sw.context_lens.sum())} cached tokens), {reps} repetitions, "
                      f"{el:.1f} s on {cores} threads (disjoint sequence slices)",
            "tokens_per_s": round(sw.num_decode * reps / el, 3)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = workload(args.workload, args.layers)
    cores = os.cpu_count() or 1
    sw, step, kv = oracle_sample(w, 64, cores)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = kv / (ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(w),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step: one layer of the first {sw.num_seqs} sequences "
                                   f"of {w.name} ({int(sw.context_lens.sum())} cached tokens), "
                                   f"on {cores} host threads (disjoint sequence slices)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def relaunch_with_torchrun(args_list, n: int) -> int:
    """`bench.py --gpus N` started as one process: run it as N ranks on this node (one per
    GPU) under torch.distributed.run, as the multi-GPU contract launches it."""
    import socket
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *args_list]
    return subprocess.call(cmd)


def main():
    args = parse_args()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(relaunch_with_torchrun(sys.argv[1:], args.gpus))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        sys.exit(2)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.kernels_only:
        import torch
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        peak, peak_src = measured_peaks()
        print(json.dumps({"reshape_and_cache": measure_store(dev, peak, peak_src),
                          "copy_blocks": measure_copy_blocks(dev, peak, peak_src)}), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    try:
        run_gpu(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
