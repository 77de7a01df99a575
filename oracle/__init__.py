"""CPU oracle for the paged KV-cache hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  The product library (``paged_kv_cache_299_gb300``) never imports
it, and it never imports the product: the two share no code.  The arithmetic lives in
``pagedkv_oracle.c`` (plain single-threaded C, double accumulation); this module only
compiles it with gcc and marshals numpy arrays through ctypes.

Every function cites the page passage it restates in the C source.  Arrays:
  * bf16 tensors are passed as ``numpy.uint16`` bit patterns;
  * tables and lengths are ``int32``; slot mappings ``int64``;
  * outputs of the attention functions are ``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()

OK, BAD_ARG, BAD_BLOCK, BAD_POSITION = 0, 1, 2, 3


def compile_source(src: str, out: str) -> str:
    """gcc the oracle source ``src`` into shared library ``out`` (no fast-math, no FMA
    contraction, so x86 and Arm hosts round identically)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle and return the library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.pko_blocks_for_tokens.argtypes = [i64, i32]
    lib.pko_blocks_for_tokens.restype = i64
    lib.pko_slot_mapping.argtypes = [P, i32, P, P, i32, i32, i32, P]
    lib.pko_slot_mapping.restype = ctypes.c_int
    lib.pko_reshape_and_cache.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P]
    lib.pko_reshape_and_cache.restype = ctypes.c_int
    lib.pko_prefill_chunk.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, P, i32, P, i32,
                                      f64]
    lib.pko_prefill_chunk.restype = ctypes.c_int
    lib.pko_decode.argtypes = [P, P, i32, P, P, i32, i32, i32, i32, P, i32, P, i32, f64]
    lib.pko_decode.restype = ctypes.c_int
    lib.pko_copy_blocks.argtypes = [P, P, i32, i32, i32, i32, P, i32]
    lib.pko_copy_blocks.restype = ctypes.c_int
    return lib


class use_library:
    """Context manager that routes every oracle call to another build of the oracle
    source (the mutation tests use it to plant a mistake and watch a pin fail)."""

    def __init__(self, path):
        self.lib = _bind(ctypes.CDLL(path))

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = self.lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = _bind(ctypes.CDLL(build()))
            _lib = lib
    return _lib


def _arr(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def blocks_for_tokens(tokens: int, block_size: int = 16) -> int:
    return int(_load().pko_blocks_for_tokens(tokens, block_size))


def slot_mapping(block_tables, context_lens, query_start_loc, num_blocks, block_size=16):
    """Return (slot_mapping int64 [T], error code)."""
    bt = _arr(block_tables, np.int32)
    cl = _arr(context_lens, np.int32)
    qsl = _arr(query_start_loc, np.int32)
    num_seqs = cl.shape[0]
    total = int(qsl[-1]) if num_seqs else 0
    out = np.empty(max(total, 1), dtype=np.int64)
    err = _load().pko_slot_mapping(_ptr(bt), bt.shape[1] if bt.ndim == 2 else 0, _ptr(cl),
                                   _ptr(qsl), num_seqs, num_blocks, block_size, _ptr(out))
    return out[:total], int(err)


def reshape_and_cache(key, value, slot_mapping_, key_cache, value_cache):
    """In-place store into key_cache / value_cache (uint16 [NB, Hkv, bs, D]); returns error."""
    k = _arr(key, np.uint16)
    v = _arr(value, np.uint16)
    sm = _arr(slot_mapping_, np.int64)
    if not (key_cache.flags.c_contiguous and value_cache.flags.c_contiguous):
        raise ValueError("caches must be contiguous")
    if key_cache.dtype != np.uint16 or value_cache.dtype != np.uint16:
        raise TypeError("caches must be uint16 bf16 bit patterns")
    nb, hkv, bs, d = key_cache.shape
    return int(_load().pko_reshape_and_cache(_ptr(k), _ptr(v), _ptr(sm), sm.shape[0], hkv, d,
                                             bs, nb, _ptr(key_cache), _ptr(value_cache)))


def decode(q, key_cache, value_cache, block_tables, context_lens, scale):
    """Return (out float64 [S, Hq, D], error code)."""
    q = _arr(q, np.uint16)
    kc = _arr(key_cache, np.uint16)
    vc = _arr(value_cache, np.uint16)
    bt = _arr(block_tables, np.int32)
    cl = _arr(context_lens, np.int32)
    s, hq, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    assert d == d2
    out = np.zeros((s, hq, d), dtype=np.float64)
    err = _load().pko_decode(_ptr(out), _ptr(q), s, _ptr(kc), _ptr(vc), nb, hkv, d, bs,
                             _ptr(bt), bt.shape[1], _ptr(cl), hq, float(scale))
    return out, int(err)


def prefill_chunk(q, query_start_loc, key_cache, value_cache, block_tables, context_lens,
                  scale):
    """Return (out float64 [Tq, Hq, D], error code)."""
    q = _arr(q, np.uint16)
    qsl = _arr(query_start_loc, np.int32)
    kc = _arr(key_cache, np.uint16)
    vc = _arr(value_cache, np.uint16)
    bt = _arr(block_tables, np.int32)
    cl = _arr(context_lens, np.int32)
    tq, hq, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    assert d == d2
    out = np.zeros((tq, hq, d), dtype=np.float64)
    err = _load().pko_prefill_chunk(_ptr(out), _ptr(q), _ptr(qsl), cl.shape[0], _ptr(kc),
                                    _ptr(vc), nb, hkv, d, bs, _ptr(bt), bt.shape[1],
                                    _ptr(cl), hq, float(scale))
    return out, int(err)


def copy_blocks(key_cache, value_cache, block_mapping):
    """In-place block copies (pairs [n, 2] of src, dst); returns the error code."""
    bm = _arr(np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2), np.int64)
    if not (key_cache.flags.c_contiguous and value_cache.flags.c_contiguous):
        raise ValueError("caches must be contiguous")
    nb, hkv, bs, d = key_cache.shape
    return int(_load().pko_copy_blocks(_ptr(key_cache), _ptr(value_cache), nb, hkv, d, bs,
                                       _ptr(bm), bm.shape[0]))
