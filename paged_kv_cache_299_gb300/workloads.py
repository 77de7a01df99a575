"""Seeded synthetic inputs for the paged KV-cache path.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle's tests.
It holds no step of the method: it only draws sequence lengths, shuffles a pool of
physical block ids into per-sequence block tables, and draws bf16 N(0, 1) values.  Slot
mappings, the scatter, the block walk and the attention are computed independently by the
library and by the oracle from these inputs.

Shapes follow Llama-3.2-1B attention as described in "tiny-vllm (1)" (geonuchoi.com):
32 query heads over hidden 2048 gives head_dim 64, and the GQA figure groups 4 query
heads per K/V head, hence 8 K/V heads.  Blocks hold 16 tokens ("vLLM", PagedAttention).

A workload is one "step": every sequence already holds ``hist_lens[s]`` cached tokens and
appends ``new_lens[s]`` tokens.  The first ``num_prefill`` sequences are prefill chunks
(every new token is a causal query row); the rest are decode sequences whose single query
is their newest token.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
BLOCK_SIZE = 16
SCALE = 0.125  # 1/sqrt(64)
NAN_BF16 = 0x7FC0  # quiet-NaN bf16 bit pattern used to poison unused pool slots


def _ceil_div(a, b):
    return -(-a // b)


def _cumsum0(x):
    out = np.zeros(len(x) + 1, dtype=np.int64)
    np.cumsum(x, out=out[1:])
    if out[-1] >= 2**31:
        raise ValueError("token count overflows int32")
    return out.astype(np.int32)


@dataclass
class Workload:
    name: str
    hist_lens: np.ndarray  # int32 [S] tokens already cached
    new_lens: np.ndarray  # int32 [S] tokens appended this step
    num_prefill: int  # leading sequences that are causal prefill chunks
    num_blocks: int  # physical blocks per pool (per layer)
    block_tables: np.ndarray  # int32 [S, max_blocks], -1 padded
    seed: int
    layers: int = 1
    big_key_fraction: float = 0.0  # share of key vectors multiplied by big_key_factor
    big_key_factor: float = 8.0
    partition_tokens: int = 0  # split-KV partition the workload asks for (0: library choice)
    num_q_heads: int = NUM_Q_HEADS
    num_kv_heads: int = NUM_KV_HEADS
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    scale: float = SCALE
    meta: dict = field(default_factory=dict)

    # ---- structure -------------------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return int(self.hist_lens.shape[0])

    @property
    def num_decode(self) -> int:
        return self.num_seqs - self.num_prefill

    @property
    def context_lens(self) -> np.ndarray:
        return (self.hist_lens + self.new_lens).astype(np.int32)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def hist_start_loc(self) -> np.ndarray:
        return _cumsum0(self.hist_lens)

    @property
    def new_start_loc(self) -> np.ndarray:
        return _cumsum0(self.new_lens)

    @property
    def prefill_query_start_loc(self) -> np.ndarray:
        return _cumsum0(self.new_lens[: self.num_prefill])

    @property
    def decode_context_lens(self) -> np.ndarray:
        return self.context_lens[self.num_prefill:]

    @property
    def decode_block_tables(self) -> np.ndarray:
        return self.block_tables[self.num_prefill:]

    def decode_kv_bytes(self) -> int:
        """Bytes of live K+V the decode attention must read (all layers)."""
        per_tok = 2 * self.num_kv_heads * self.head_dim * 2
        return int(self.decode_context_lens.astype(np.int64).sum()) * per_tok * self.layers

    # ---- values ----------------------------------------------------------------------
    def values(self, layer: int = 0, device="cpu") -> dict:
        """bf16 tensors for one layer, drawn from a generator seeded by (seed, layer).

        hist_k / hist_v: [sum(hist_lens), Hkv, D], sequence-major, position order;
        new_k / new_v:   [sum(new_lens), Hkv, D];
        q_prefill:       [sum(new_lens[:num_prefill]), Hq, D] (one row per chunk token);
        q_decode:        [num_decode, Hq, D] (query of each decode sequence's newest token).
        """
        dev = torch.device(device)
        g = torch.Generator(device=dev)
        g.manual_seed(int(self.seed) * 1009 + int(layer))
        hq, hkv, d = self.num_q_heads, self.num_kv_heads, self.head_dim
        n_hist = int(self.hist_lens.sum())
        n_new = int(self.new_lens.sum())
        n_pre = int(self.new_lens[: self.num_prefill].sum())

        def normal(*shape):
            x = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
            return x.to(torch.bfloat16)

        out = {
            "hist_k": normal(n_hist, hkv, d),
            "hist_v": normal(n_hist, hkv, d),
            "new_k": normal(n_new, hkv, d),
            "new_v": normal(n_new, hkv, d),
            "q_prefill": normal(n_pre, hq, d),
            "q_decode": normal(self.num_decode, hq, d),
        }
        if self.big_key_fraction > 0:
            for name, n in (("hist_k", n_hist), ("new_k", n_new)):
                pick = torch.rand(n, hkv, 1, generator=g, device=dev) < self.big_key_fraction
                big = out[name] * torch.tensor(self.big_key_factor, dtype=torch.bfloat16,
                                               device=dev)
                out[name] = torch.where(pick, big, out[name])
        return out


def make_workload(name, hist_lens, new_lens, num_prefill=0, seed=0, pool_slack=0.10,
                  pool_blocks=None, layers=1, **kw) -> Workload:
    """Shuffle a pool of physical blocks and draw each sequence's table from it.

    The pool holds ``ceil((1 + pool_slack) * total_blocks)`` blocks unless ``pool_blocks``
    is given; block ids are a seeded permutation and each sequence takes the next ids
    without replacement, so tables are non-contiguous and disjoint.
    """
    hist_lens = np.asarray(hist_lens, dtype=np.int32)
    new_lens = np.asarray(new_lens, dtype=np.int32)
    if hist_lens.shape != new_lens.shape:
        raise ValueError("hist_lens and new_lens differ in shape")
    ctx = hist_lens.astype(np.int64) + new_lens
    need = _ceil_div(ctx, BLOCK_SIZE).astype(np.int64)
    total = int(need.sum())
    if pool_blocks is None:
        pool_blocks = max(1, int(np.ceil(total * (1.0 + pool_slack))))
    if pool_blocks < total:
        raise ValueError("pool smaller than the blocks the sequences need")
    rng = np.random.default_rng(seed)
    perm = rng.permutation(pool_blocks).astype(np.int32)
    max_blocks = max(1, int(need.max()) if len(need) else 1)
    tables = np.full((len(ctx), max_blocks), -1, dtype=np.int32)
    cursor = 0
    for s, n in enumerate(need):
        tables[s, :n] = perm[cursor:cursor + n]
        cursor += n
    return Workload(name=name, hist_lens=hist_lens, new_lens=new_lens,
                    num_prefill=int(num_prefill), num_blocks=int(pool_blocks),
                    block_tables=tables, seed=int(seed), layers=int(layers), **kw)


# ---- the five workloads of the benchmark and the parity tests --------------------------

def single_sequence_300(seed=1001) -> Workload:
    """One sequence of 300 tokens (19 blocks) at a seeded permutation of a 64-block pool;
    all 300 tokens are stored this step, then one decode query attends them."""
    return make_workload("single_seq_300", [0], [300], seed=seed, pool_blocks=64)


def decode_batch64_uniform(seed=1002) -> Workload:
    """Decode batch 64, contexts uniform in [128, 2048], pool = blocks needed + 10%."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(128, 2048, size=64, endpoint=True)
    return make_workload("decode_b64_u128_2048", ctx - 1, np.ones(64, np.int32),
                         seed=seed)


def decode_batch256_lognormal(seed=1003, layers=16) -> Workload:
    """Decode batch 256, contexts lognormal (median 1024, sigma 0.8) clipped to [1, 8192],
    16 layers of pools resident (one pool per layer, shared block tables)."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(256)
    ctx = np.clip(np.round(np.exp(np.log(1024.0) + 0.8 * z)), 1, 8192).astype(np.int32)
    return make_workload("decode_b256_lognormal_16L", ctx - 1, np.ones(256, np.int32),
                         seed=seed, layers=layers)


def long_context_batch4(seed=1004) -> Workload:
    """Long-context decode: 4 sequences of 131072 tokens, 1% of key vectors x8,
    split-KV partitions of 512 tokens."""
    ctx = np.full(4, 131072, dtype=np.int32)
    return make_workload("decode_b4_131072", ctx - 1, np.ones(4, np.int32), seed=seed,
                         big_key_fraction=0.01, partition_tokens=512)


def mixed_prefill_decode(seed=1005) -> Workload:
    """Mixed step: 8 prefill sequences append a 512-token causal chunk over 0..2048 prior
    tokens; 248 decode sequences with contexts uniform in [1, 4096]."""
    rng = np.random.default_rng(seed)
    prior = rng.integers(0, 2048, size=8, endpoint=True)
    dctx = rng.integers(1, 4096, size=248, endpoint=True)
    hist = np.concatenate([prior, dctx - 1])
    new = np.concatenate([np.full(8, 512), np.ones(248)])
    return make_workload("mixed_8x512_prefill_248_decode", hist, new, num_prefill=8,
                         seed=seed)


# by the short names bench.py takes (--workload)
WORKLOADS = {"single_seq_300": single_sequence_300, "decode_b64": decode_batch64_uniform,
             "decode_b256": decode_batch256_lognormal, "long_context_b4": long_context_batch4,
             "mixed_step": mixed_prefill_decode}


def random_small(seed, num_seqs=3, max_ctx=64, num_prefill=0, max_chunk=40,
                 pool_slack=0.5, **kw) -> Workload:
    """Small ragged workload for sweeps: random contexts, random chunk lengths."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1, max_ctx, size=num_seqs, endpoint=True)
    new = np.ones(num_seqs, dtype=np.int64)
    for s in range(num_prefill):
        new[s] = rng.integers(1, min(max_chunk, ctx[s]), endpoint=True)
    return make_workload(f"random_{seed}", ctx - new, new, num_prefill=num_prefill,
                         seed=seed, pool_slack=pool_slack, **kw)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def nan_pool(num_blocks, num_kv_heads=NUM_KV_HEADS, block_size=BLOCK_SIZE,
             head_dim=HEAD_DIM) -> np.ndarray:
    """Host pool of bf16 NaN bit patterns, [NB, Hkv, block, D]."""
    return np.full((num_blocks, num_kv_heads, block_size, head_dim), NAN_BF16,
                   dtype=np.uint16)
