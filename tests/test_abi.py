"""The C-ABI library builds for sm_103a, loads, exports every symbol the header declares,
and rejects bad arguments on the host (these calls return before any CUDA call, so they
run without a GPU)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_299_gb300 import binding as pa
from paged_kv_cache_299_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_library_builds_and_exports_every_declared_symbol():
    lib = pa.load()
    names = declared_functions()
    assert set(names) == set(pa.EXPORTED)
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings():
    lib = pa.load()
    for code in range(-7, 1):
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(-99) == b"unknown status"


def _desc(nb=4, hkv=8, d=64, bs=16):
    return pa.CacheDesc(nb, hkv, d, bs)


def test_host_rejects_bad_arguments_without_touching_the_device():
    lib = pa.load()
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails its host checks first
    # unsupported head_dim / block_size
    assert lib.pa_reshape_and_cache(fake, fake, fake, 1, fake, fake, _desc(d=128), None,
                                    None) == pa.PA_ERR_UNSUPPORTED
    assert b"head_dim" in lib.pa_last_error()
    assert lib.pa_reshape_and_cache(fake, fake, fake, 1, fake, fake, _desc(bs=32), None,
                                    None) == pa.PA_ERR_UNSUPPORTED
    # null pointers, misalignment, negative sizes
    assert lib.pa_reshape_and_cache(None, fake, fake, 1, fake, fake, _desc(), None,
                                    None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(P(0x1008), fake, fake, 1, fake, fake, _desc(), None,
                                    None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(fake, fake, fake, -1, fake, fake, _desc(), None,
                                    None) == pa.PA_ERR_INVALID_ARG
    # empty calls succeed without launching
    assert lib.pa_reshape_and_cache(None, None, None, 0, None, None, _desc(), None,
                                    None) == pa.PA_OK
    assert lib.pa_compute_slot_mapping(None, 1, None, None, 0, 0, _desc(), None, None,
                                       None) == pa.PA_OK
    assert lib.pa_compute_slot_mapping(fake, 1, fake, None, 2, 3, _desc(), fake, None,
                                       None) == pa.PA_ERR_INVALID_ARG
    # decode: group of 3 unsupported, partition not a multiple of 16, too many sequences
    args = [fake, fake, fake, fake, _desc(), fake, 4, fake]
    assert lib.pa_decode(*args, 2, 24, ctypes.c_float(0.125), 64, 0, fake, 1 << 20, 0, None,
                         None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode(*args, 2, 32, ctypes.c_float(0.125), 64, 24, fake, 1 << 20, 0, None,
                         None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode(*args, 5000, 32, ctypes.c_float(0.125), 64, 0, fake, 1 << 20, 0, None,
                         None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode(*args, 0, 32, ctypes.c_float(0.125), 64, 0, None, 0, 0, None,
                         None) == pa.PA_OK
    assert lib.pa_decode(*args, 2, 32, ctypes.c_float(-1.0), 64, 0, fake, 1 << 20, 0, None,
                         None) == pa.PA_ERR_INVALID_ARG
    # pools beyond 2^31 rows of 64 head dims are refused by the attention calls
    big = pa.CacheDesc(1 << 24, 8, 64, 16)  # 2^24 blocks x 8 heads x 16 rows = 2^31 rows
    assert lib.pa_decode(fake, fake, fake, fake, big, fake, 4, fake, 2, 32,
                         ctypes.c_float(0.125), 64, 0, fake, 1 << 20, 0, None,
                         None) == pa.PA_ERR_UNSUPPORTED
    assert b"2^31" in lib.pa_last_error()
    # launch flags: unknown bits are rejected before any launch, with or without an SM budget
    # (bits 16-31), and by the chunk call too
    for flags in (2, 4 | pa.PA_LAUNCH_MAX_SMS(8), 0x8000):
        assert lib.pa_decode(*args, 2, 32, ctypes.c_float(0.125), 64, 0, fake, 1 << 20, flags,
                             None, None) == pa.PA_ERR_INVALID_ARG
        assert b"launch flags" in lib.pa_last_error()
        assert lib.pa_prefill_chunk_ex(fake, fake, fake, 16, 8, fake, fake, _desc(), fake, 4,
                                       fake, 2, 32, ctypes.c_float(0.125), flags, None,
                                       None) == pa.PA_ERR_INVALID_ARG
        assert b"launch flags" in lib.pa_last_error()
    # the chunk call's own checks come first, as in pa_prefill_chunk
    assert lib.pa_prefill_chunk_ex(fake, fake, fake, 16, 8, fake, fake, _desc(), fake, 4, fake,
                                   2, 8, ctypes.c_float(0.125), 0, None,
                                   None) == pa.PA_ERR_UNSUPPORTED
    # prefill needs group 4
    assert lib.pa_prefill_chunk(fake, fake, fake, 16, 8, fake, fake, _desc(), fake, 4, fake, 2,
                                8, ctypes.c_float(0.125), None, None) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_prefill_chunk(fake, fake, fake, 4, 8, fake, fake, _desc(), fake, 4, fake, 2,
                                32, ctypes.c_float(0.125), None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_workspace_size(2, 8, 24, 64, 0) == 0
    assert lib.pa_check_device_status(None, None) == pa.PA_ERR_INVALID_ARG
    # stream read: null, misaligned, size not a multiple of 16
    assert lib.pa_stream_read(None, 64, fake, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_stream_read(P(0x1008), 64, fake, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_stream_read(fake, 24, fake, None) == pa.PA_ERR_INVALID_ARG


def test_build_targets_sm103a_only():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(build.build())


def test_varlen_workspace_size_and_host_checks():
    """The varlen workspace is the decode kernel's (its one-row sequences run there): its
    size comes from the decode plan on the current device, so without a GPU the query
    returns 0, except for the sizes that need no device (no sequences: 16 bytes; more than
    the decode kernel's 4096 sequences: 16 bytes, every row then runs on the chunk kernel).
    Missing or misaligned workspaces are refused before any device query."""
    import torch
    lib = pa.load()
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert lib.pa_varlen_workspace_size(-1, 4) == 0
    assert lib.pa_varlen_workspace_size(0, 0) == 16
    assert lib.pa_varlen_workspace_size(5000, 5000) == 16
    if not torch.cuda.is_available():
        assert lib.pa_varlen_workspace_size(256, 4344) == 0
    args = [fake, fake, fake, 40, 32, fake, fake, _desc(), fake, 4, fake, 2, 32,
            ctypes.c_float(0.125)]
    assert lib.pa_attention_varlen(*args, None, 1 << 20, None, None) == pa.PA_ERR_WORKSPACE
    assert lib.pa_attention_varlen(*args, P(0x1008), 1 << 20, None, None) == pa.PA_ERR_WORKSPACE
    assert b"workspace" in lib.pa_last_error()
    # the checks shared with pa_prefill_chunk come first
    bad = list(args)
    bad[12] = 24  # group of 3
    assert lib.pa_attention_varlen(*bad, fake, 1 << 20, None, None) == pa.PA_ERR_UNSUPPORTED
    bad = list(args)
    bad[4] = 41  # max_query_len > num_query_tokens
    assert lib.pa_attention_varlen(*bad, fake, 1 << 20, None, None) == pa.PA_ERR_INVALID_ARG
    # an empty batch needs no workspace and launches nothing
    empty = list(args)
    empty[11] = 0
    assert lib.pa_attention_varlen(*empty, None, 0, None, None) == pa.PA_OK


def test_static_scratch_size_matches_the_header():
    text = open(HEADER).read()
    m = re.search(r"#define PA_DECODE_STATIC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m, "PA_DECODE_STATIC_SCRATCH_BYTES not found in the header"
    assert int(m.group(1)) << int(m.group(2)) == pa.PA_DECODE_STATIC_SCRATCH_BYTES


def test_launch_flags_match_the_header():
    text = open(HEADER).read()
    for name in ("PA_LAUNCH_DEFAULT", "PA_LAUNCH_OVERLAP_PREVIOUS"):
        m = re.search(r"#define %s (\d+)u" % name, text)
        assert m, name + " not found in the header"
        assert int(m.group(1)) == getattr(pa, name)
    m = re.search(r"#define PA_LAUNCH_MAX_SMS\(n\) \(\(uint32_t\)\(n\) << (\d+)\)", text)
    assert m, "PA_LAUNCH_MAX_SMS not found in the header"
    assert pa.PA_LAUNCH_MAX_SMS(88) == 88 << int(m.group(1))
    for bad in (0, 1 << 16):
        with pytest.raises(ValueError):
            pa.PA_LAUNCH_MAX_SMS(bad)
