"""Python binding of libpagedkv.so: the C-ABI calls of include/pagedkv.h under the same
names, taking torch CUDA tensors.

This module only marshals arguments (dtype / shape / device checks, data pointers, the
current CUDA stream) and raises ``PagedKVError`` on a non-OK status; every step of the
path runs in the library's kernels.  There is no fallback: if the library is missing or
fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32)]


PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_WORKSPACE = -4
PA_ERR_DEVICE_INDEX = -5
PA_ERR_DEVICE_TIMEOUT = -6
PA_ERR_OUT_OF_BLOCKS = -7
DEVFLAG_BAD_BLOCK, DEVFLAG_BAD_SLOT, DEVFLAG_BAD_CONTEXT, DEVFLAG_TIMEOUT = 1, 2, 4, 8
# Size of the library-owned device scratch of pa_decode_static_scratch (bytes).
PA_DECODE_STATIC_SCRATCH_BYTES = 8 << 20
# Launch flags of pa_decode / pa_decode_append (include/pagedkv.h states the contract).
PA_LAUNCH_DEFAULT = 0
PA_LAUNCH_OVERLAP_PREVIOUS = 1


def PA_LAUNCH_MAX_SMS(n: int) -> int:
    """Launch-flag bits confining a persistent grid to at most n SMs (1 .. 65535)."""
    if not 1 <= int(n) <= 0xFFFF:
        raise ValueError(f"PA_LAUNCH_MAX_SMS: n = {n} outside 1 .. 65535")
    return int(n) << 16

# Every symbol include/pagedkv.h declares.
EXPORTED = ("pa_compute_slot_mapping", "pa_reshape_and_cache", "pa_decode_workspace_size",
            "pa_decode", "pa_prefill_chunk", "pa_check_device_status", "pa_status_string",
            "pa_last_error", "pa_decode_static_scratch", "pa_copy_blocks", "pa_bm_create",
            "pa_bm_destroy", "pa_bm_num_free_blocks", "pa_bm_ref_count", "pa_bm_add_sequence",
            "pa_bm_fork", "pa_bm_append_tokens", "pa_bm_free_sequence", "pa_bm_num_tokens",
            "pa_bm_block_table", "pa_decode_append", "pa_selftest_wait_timeout",
            "pa_varlen_workspace_size", "pa_attention_varlen", "pa_stream_read",
            "pa_prefill_chunk_ex", "pa_attention_varlen_ex")


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load (building first if the sources are newer) and bind the library."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    if path is None:
        path = _build.build()
    if not os.path.exists(path):
        raise PagedKVError(PA_ERR_CUDA, f"libpagedkv.so not found at {path}")
    lib = ctypes.CDLL(path)
    P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    st = ctypes.c_int
    lib.pa_compute_slot_mapping.argtypes = [P, i32, P, P, i32, i32, CacheDesc, P, P, P]
    lib.pa_compute_slot_mapping.restype = st
    lib.pa_reshape_and_cache.argtypes = [P, P, P, i32, P, P, CacheDesc, P, P]
    lib.pa_reshape_and_cache.restype = st
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.pa_decode_workspace_size.restype = sz
    u32 = ctypes.c_uint32
    lib.pa_decode.argtypes = [P, P, P, P, CacheDesc, P, i32, P, i32, i32, f32, i32, i32, P, sz,
                              u32, P, P]
    lib.pa_decode.restype = st
    lib.pa_prefill_chunk.argtypes = [P, P, P, i32, i32, P, P, CacheDesc, P, i32, P, i32, i32,
                                     f32, P, P]
    lib.pa_prefill_chunk.restype = st
    lib.pa_prefill_chunk_ex.argtypes = [P, P, P, i32, i32, P, P, CacheDesc, P, i32, P, i32, i32,
                                        f32, u32, P, P]
    lib.pa_prefill_chunk_ex.restype = st
    lib.pa_varlen_workspace_size.argtypes = [i32, i32]
    lib.pa_varlen_workspace_size.restype = sz
    lib.pa_attention_varlen.argtypes = [P, P, P, i32, i32, P, P, CacheDesc, P, i32, P, i32,
                                        i32, f32, P, sz, P, P]
    lib.pa_attention_varlen.restype = st
    lib.pa_attention_varlen_ex.argtypes = [P, P, P, i32, i32, P, P, CacheDesc, P, i32, P, i32,
                                           i32, f32, P, sz, u32, P, P]
    lib.pa_attention_varlen_ex.restype = st
    lib.pa_decode_static_scratch.argtypes = [P, P, P, P, CacheDesc, P, i32, P, i32, i32, f32,
                                             i32, i32, P, P]
    lib.pa_decode_static_scratch.restype = st
    lib.pa_decode_append.argtypes = [P, P, P, P, P, P, CacheDesc, P, i32, P, i32, i32, f32, i32,
                                     i32, P, sz, u32, P, P]
    lib.pa_decode_append.restype = st
    lib.pa_copy_blocks.argtypes = [P, P, CacheDesc, P, i32, P, P]
    lib.pa_copy_blocks.restype = st
    i64 = ctypes.c_int64
    lib.pa_bm_create.argtypes = [i32, i32, ctypes.POINTER(P)]
    lib.pa_bm_create.restype = st
    lib.pa_bm_destroy.argtypes = [P]
    lib.pa_bm_destroy.restype = None
    lib.pa_bm_num_free_blocks.argtypes = [P]
    lib.pa_bm_num_free_blocks.restype = i32
    lib.pa_bm_ref_count.argtypes = [P, i32]
    lib.pa_bm_ref_count.restype = i32
    lib.pa_bm_add_sequence.argtypes = [P, i64]
    lib.pa_bm_add_sequence.restype = st
    lib.pa_bm_fork.argtypes = [P, i64, i64]
    lib.pa_bm_fork.restype = st
    lib.pa_bm_append_tokens.argtypes = [P, i64, i32, P, i32, ctypes.POINTER(i32)]
    lib.pa_bm_append_tokens.restype = st
    lib.pa_bm_free_sequence.argtypes = [P, i64]
    lib.pa_bm_free_sequence.restype = st
    lib.pa_bm_num_tokens.argtypes = [P, i64]
    lib.pa_bm_num_tokens.restype = i64
    lib.pa_bm_block_table.argtypes = [P, i64, P, i32]
    lib.pa_bm_block_table.restype = i32
    lib.pa_selftest_wait_timeout.argtypes = [P, i32, P]
    lib.pa_selftest_wait_timeout.restype = st
    lib.pa_stream_read.argtypes = [P, sz, P, P]
    lib.pa_stream_read.restype = st
    lib.pa_check_device_status.argtypes = [P, P]
    lib.pa_check_device_status.restype = st
    lib.pa_status_string.argtypes = [st]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_error.argtypes = []
    lib.pa_last_error.restype = ctypes.c_char_p
    if path == _build.LIB:
        _lib = lib
    return lib


def _check(status: int, what: str):
    if status != PA_OK:
        lib = load()
        msg = lib.pa_last_error().decode()
        name = lib.pa_status_string(status).decode()
        raise PagedKVError(status, f"{what}: {name} ({msg})")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def cache_desc(key_cache: torch.Tensor) -> CacheDesc:
    nb, hkv, bs, d = key_cache.shape
    return CacheDesc(nb, hkv, d, bs)


def new_device_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def pa_compute_slot_mapping(block_tables, context_lens, query_start_loc, num_tokens,
                            key_cache, slot_mapping=None, device_status=None, stream=None):
    """int64 slot of every appended token (see include/pagedkv.h)."""
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if query_start_loc is not None:
        _need(query_start_loc, "query_start_loc", torch.int32, 1)
    if slot_mapping is None:
        slot_mapping = torch.empty(num_tokens, dtype=torch.int64, device=block_tables.device)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    st = load().pa_compute_slot_mapping(
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), _ptr(query_start_loc),
        context_lens.shape[0], int(num_tokens), cache_desc(key_cache), _ptr(slot_mapping),
        _ptr(device_status), _stream(stream))
    _check(st, "pa_compute_slot_mapping")
    return slot_mapping


def pa_reshape_and_cache(key, value, slot_mapping, key_cache, value_cache, device_status=None,
                         stream=None):
    """Store key/value [T, Hkv, D] into the paged pools at slot_mapping[T]."""
    _need(key, "key", torch.bfloat16, 3)
    _need(value, "value", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    _need(value_cache, "value_cache", torch.bfloat16, 4)
    if key.shape != value.shape or key_cache.shape != value_cache.shape:
        raise ValueError("key/value or cache shapes differ")
    if key.shape[0] != slot_mapping.shape[0] or key.shape[1:] != (key_cache.shape[1],
                                                                   key_cache.shape[3]):
        raise ValueError("key shape does not match slot_mapping / cache")
    st = load().pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(slot_mapping), key.shape[0],
                                     _ptr(key_cache), _ptr(value_cache), cache_desc(key_cache),
                                     _ptr(device_status), _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_decode_workspace_size(num_seqs, num_kv_heads, num_q_heads, max_context_len,
                             partition_tokens=0) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_kv_heads, num_q_heads,
                                               max_context_len, partition_tokens))


def pa_decode(out, q, key_cache, value_cache, block_tables, context_lens, scale,
              max_context_len, partition_tokens=0, workspace=None, device_status=None,
              stream=None, launch_flags=PA_LAUNCH_DEFAULT):
    """Paged decode attention; writes out [S, Hq, D] (bf16).  launch_flags: see
    PA_LAUNCH_OVERLAP_PREVIOUS in include/pagedkv.h."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    _need(value_cache, "value_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    num_seqs, hq, _ = q.shape
    if out.shape != q.shape or block_tables.shape[0] != num_seqs or \
            context_lens.shape[0] != num_seqs:
        raise ValueError("q/out/block_tables/context_lens disagree on the sequence count")
    if workspace is None:
        need = pa_decode_workspace_size(num_seqs, key_cache.shape[1], hq, max_context_len,
                                        partition_tokens)
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    st = load().pa_decode(_ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache),
                          cache_desc(key_cache), _ptr(block_tables), block_tables.shape[1],
                          _ptr(context_lens), num_seqs, hq, float(scale), int(max_context_len),
                          int(partition_tokens), _ptr(workspace), workspace.numel(),
                          int(launch_flags), _ptr(device_status), _stream(stream))
    _check(st, "pa_decode")
    return out


def pa_decode_append(out, q, key, value, key_cache, value_cache, block_tables, context_lens,
                     scale, max_context_len, partition_tokens=0, workspace=None,
                     device_status=None, stream=None, launch_flags=PA_LAUNCH_DEFAULT):
    """Store each sequence's newest token (key/value [S, Hkv, D]) and run paged decode
    attention, in one launch; bit-identical to pa_reshape_and_cache + pa_decode.
    launch_flags: see PA_LAUNCH_OVERLAP_PREVIOUS in include/pagedkv.h."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(key, "key", torch.bfloat16, 3)
    _need(value, "value", torch.bfloat16, 3)
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    _need(value_cache, "value_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    num_seqs, hq, _ = q.shape
    if out.shape != q.shape or key.shape != value.shape or key.shape[0] != num_seqs or \
            key.shape[1:] != (key_cache.shape[1], key_cache.shape[3]) or \
            block_tables.shape[0] != num_seqs or context_lens.shape[0] != num_seqs:
        raise ValueError("pa_decode_append argument shapes disagree")
    if workspace is None:
        need = pa_decode_workspace_size(num_seqs, key_cache.shape[1], hq, max_context_len,
                                        partition_tokens)
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    st = load().pa_decode_append(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(key_cache),
                                 _ptr(value_cache), cache_desc(key_cache), _ptr(block_tables),
                                 block_tables.shape[1], _ptr(context_lens), num_seqs, hq,
                                 float(scale), int(max_context_len), int(partition_tokens),
                                 _ptr(workspace), workspace.numel(), int(launch_flags),
                                 _ptr(device_status), _stream(stream))
    _check(st, "pa_decode_append")
    return out


def pa_decode_static_scratch(out, q, key_cache, value_cache, block_tables, context_lens, scale,
                             max_context_len, partition_tokens=0, device_status=None,
                             stream=None):
    """Paged decode attention without a workspace argument: for callers that cannot
    allocate device memory, the library uses its own fixed device scratch (see
    include/pagedkv.h for the size limit and the rules on overlapping calls)."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    _need(value_cache, "value_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    num_seqs, hq, _ = q.shape
    if out.shape != q.shape or block_tables.shape[0] != num_seqs or \
            context_lens.shape[0] != num_seqs:
        raise ValueError("q/out/block_tables/context_lens disagree on the sequence count")
    st = load().pa_decode_static_scratch(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), cache_desc(key_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), num_seqs, hq,
        float(scale), int(max_context_len), int(partition_tokens), _ptr(device_status),
        _stream(stream))
    _check(st, "pa_decode_static_scratch")
    return out


def pa_prefill_chunk(out, q, query_start_loc, max_query_len, key_cache, value_cache,
                     block_tables, context_lens, scale, device_status=None, stream=None,
                     launch_flags=PA_LAUNCH_DEFAULT):
    """Causal chunked-prefill attention; writes out [Tq, Hq, D] (bf16).  launch_flags (see
    PA_LAUNCH_OVERLAP_PREVIOUS and PA_LAUNCH_MAX_SMS in include/pagedkv.h) go through
    pa_prefill_chunk_ex."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    _need(value_cache, "value_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    num_seqs = context_lens.shape[0]
    if out.shape != q.shape or query_start_loc.shape[0] != num_seqs + 1 or \
            block_tables.shape[0] != num_seqs:
        raise ValueError("prefill argument shapes disagree")
    args = (_ptr(out), _ptr(q), _ptr(query_start_loc), q.shape[0], int(max_query_len),
            _ptr(key_cache), _ptr(value_cache), cache_desc(key_cache), _ptr(block_tables),
            block_tables.shape[1], _ptr(context_lens), num_seqs, q.shape[1], float(scale))
    if launch_flags == PA_LAUNCH_DEFAULT:
        st = load().pa_prefill_chunk(*args, _ptr(device_status), _stream(stream))
        _check(st, "pa_prefill_chunk")
    else:
        st = load().pa_prefill_chunk_ex(*args, int(launch_flags), _ptr(device_status),
                                        _stream(stream))
        _check(st, "pa_prefill_chunk_ex")
    return out


def pa_varlen_workspace_size(num_seqs, num_query_tokens) -> int:
    return int(load().pa_varlen_workspace_size(num_seqs, num_query_tokens))


def pa_attention_varlen(out, q, query_start_loc, max_query_len, key_cache, value_cache,
                        block_tables, context_lens, scale, workspace=None, device_status=None,
                        stream=None, launch_flags=PA_LAUNCH_DEFAULT):
    """One continuous-batching step's attention (decode rows and causal chunks mixed): decode
    rows on the decode kernel, chunks on the tensor-core chunk kernel; chunk rows equal
    pa_prefill_chunk's bit for bit, decode rows pa_decode's up to rounding.  launch_flags:
    PA_LAUNCH_MAX_SMS(n) runs the decode rows on n SMs beside the chunks (through
    pa_attention_varlen_ex)."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    _need(value_cache, "value_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    num_seqs = context_lens.shape[0]
    if out.shape != q.shape or query_start_loc.shape[0] != num_seqs + 1 or \
            block_tables.shape[0] != num_seqs:
        raise ValueError("varlen argument shapes disagree")
    if workspace is None:
        workspace = torch.empty(max(16, pa_varlen_workspace_size(num_seqs, q.shape[0])),
                                dtype=torch.uint8, device=q.device)
    args = (_ptr(out), _ptr(q), _ptr(query_start_loc), q.shape[0], int(max_query_len),
            _ptr(key_cache), _ptr(value_cache), cache_desc(key_cache), _ptr(block_tables),
            block_tables.shape[1], _ptr(context_lens), num_seqs, q.shape[1], float(scale),
            _ptr(workspace), workspace.numel() * workspace.element_size())
    if launch_flags == PA_LAUNCH_DEFAULT:
        st = load().pa_attention_varlen(*args, _ptr(device_status), _stream(stream))
        _check(st, "pa_attention_varlen")
    else:
        st = load().pa_attention_varlen_ex(*args, int(launch_flags), _ptr(device_status),
                                           _stream(stream))
        _check(st, "pa_attention_varlen_ex")
    return out


def pa_check_device_status(device_status, stream=None) -> int:
    """Synchronise and translate the device status word; returns the pa_status code."""
    _need(device_status, "device_status", torch.int32, 1)
    return int(load().pa_check_device_status(_ptr(device_status), _stream(stream)))


def pa_copy_blocks(key_cache, value_cache, block_mapping, device_status=None, stream=None):
    """Copy whole physical blocks of both pools: block_mapping int64 [n, 2] (src, dst)."""
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    _need(value_cache, "value_cache", torch.bfloat16, 4)
    _need(block_mapping, "block_mapping", torch.int64, 2)
    if key_cache.shape != value_cache.shape or block_mapping.shape[1] != 2:
        raise ValueError("cache shapes differ or block_mapping is not [n, 2]")
    st = load().pa_copy_blocks(_ptr(key_cache), _ptr(value_cache), cache_desc(key_cache),
                               _ptr(block_mapping), block_mapping.shape[0], _ptr(device_status),
                               _stream(stream))
    _check(st, "pa_copy_blocks")


class BlockManager:
    """Host-side block manager of include/pagedkv.h (pa_bm_*): block tables grown on
    demand, forks that share blocks, copy-on-write pairs for pa_copy_blocks."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.pa_bm_create(num_blocks, block_size, ctypes.byref(h)), "pa_bm_create")
        self._h = h

    def close(self):
        if self._h:
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_free_blocks(self) -> int:
        return int(self._lib.pa_bm_num_free_blocks(self._h))

    def ref_count(self, block: int) -> int:
        return int(self._lib.pa_bm_ref_count(self._h, block))

    def add_sequence(self, seq_id: int):
        _check(self._lib.pa_bm_add_sequence(self._h, seq_id), "pa_bm_add_sequence")

    def fork(self, parent: int, child: int):
        _check(self._lib.pa_bm_fork(self._h, parent, child), "pa_bm_fork")

    def append_tokens(self, seq_id: int, num_tokens: int):
        """Returns the list of (src, dst) copy-on-write pairs (at most one)."""
        pairs = (ctypes.c_int64 * 2)()
        n = ctypes.c_int32(0)
        _check(self._lib.pa_bm_append_tokens(self._h, seq_id, num_tokens, pairs, 1,
                                             ctypes.byref(n)), "pa_bm_append_tokens")
        return [(int(pairs[0]), int(pairs[1]))] if n.value else []

    def free_sequence(self, seq_id: int):
        _check(self._lib.pa_bm_free_sequence(self._h, seq_id), "pa_bm_free_sequence")

    def num_tokens(self, seq_id: int) -> int:
        return int(self._lib.pa_bm_num_tokens(self._h, seq_id))

    def block_table(self, seq_id: int, max_blocks: int):
        out = (ctypes.c_int32 * max(max_blocks, 1))()
        n = int(self._lib.pa_bm_block_table(self._h, seq_id, out, max_blocks))
        if n < 0:
            _check(n, "pa_bm_block_table")
        return [int(out[i]) for i in range(max_blocks)], n


def pa_stream_read(buf, xor_out, stream=None):
    """Read every byte of `buf` once (the in-run read-bandwidth reference) and XOR its 32-bit
    words into xor_out (int32 [1] on the device, zeroed by the caller); see
    include/pagedkv.h."""
    if not buf.is_contiguous() or buf.device.type != "cuda":
        raise ValueError("buf must be a contiguous CUDA tensor")
    _need(xor_out, "xor_out", torch.int32, 1)
    nbytes = buf.numel() * buf.element_size()
    _check(load().pa_stream_read(_ptr(buf), nbytes, _ptr(xor_out), _stream(stream)),
           "pa_stream_read")
    return xor_out


def pa_selftest_wait_timeout(device_status, limit_ms=50, stream=None):
    """Launch the bounded-wait diagnostic (see include/pagedkv.h)."""
    _need(device_status, "device_status", torch.int32, 1)
    _check(load().pa_selftest_wait_timeout(_ptr(device_status), int(limit_ms), _stream(stream)),
           "pa_selftest_wait_timeout")
