"""The C-ABI library: it builds, loads without a GPU, exports every symbol the
public headers declare, and rejects bad arguments on the host before any
launch (CPU only: no compute call is made)."""

import ctypes
import glob
import os
import re

import numpy as np
import pytest

import paged_kv_cache_46_gb300 as ts
from paged_kv_cache_46_gb300 import build as ts_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ts_build.build()
    return ts.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"^TS_API\s+[\w\s\*]+?\b(ts_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def _declared_arity():
    """Parameter count of every ts_* function the public headers declare."""
    arity = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^TS_API\s+[\w\s\*]+?\b(ts_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M):
            params = m.group(2).strip()
            arity[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return arity


def test_binding_signatures_match_the_header():
    """Every function the Python binding declares has the header's parameter
    count (a mismatch would pass arguments into the wrong slots)."""
    arity = _declared_arity()
    assert len(arity) >= 13
    for name, (_, args) in ts._SIGNATURES.items():
        assert name in arity, f"{name} bound but not declared in include/"
        assert len(args) == arity[name], f"{name}: binding has {len(args)} parameters, header {arity[name]}"


def test_status_strings(lib):
    assert lib.ts_status_string(0) == b"TS_OK"
    assert lib.ts_status_string(1) == b"TS_ERR_INVALID_ARG"
    assert lib.ts_status_string(99) == b"TS_ERR_UNKNOWN"
    assert b"sm_103a" in lib.ts_version()


def test_host_validation_rejects_bad_arguments(lib):
    f = lib.ts_paged_decode_attn
    vp = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # H_q not a multiple of H_kv
    st = f(vp, vp, vp, vp, 4, vp, 2, 6, 4, 64, 16, 8, 1.0, 1, vp, None, vp, 1 << 20, None)
    assert st == ts.TS_ERR_INVALID_ARG
    assert b"multiple" in lib.ts_last_error_detail()
    # negative batch
    st = f(vp, vp, vp, vp, 4, vp, -1, 8, 2, 64, 16, 8, 1.0, 1, vp, None, vp, 1 << 20, None)
    assert st == ts.TS_ERR_INVALID_ARG
    # bad dtype
    st = f(vp, vp, vp, vp, 4, vp, 2, 8, 2, 64, 16, 8, 1.0, 7, vp, None, vp, 1 << 20, None)
    assert st == ts.TS_ERR_INVALID_ARG
    # non-finite scale
    st = f(vp, vp, vp, vp, 4, vp, 2, 8, 2, 64, 16, 8, float("nan"), 1, vp, None, vp, 1 << 20, None)
    assert st == ts.TS_ERR_INVALID_ARG
    # empty batch is a no-op
    st = f(None, None, None, None, 4, None, 0, 8, 2, 64, 16, 8, 1.0, 1, None, None, None, 0, None)
    assert st == ts.TS_OK
    # append and merge: empty batches are no-ops, bad sizes are rejected
    assert lib.ts_kv_append(None, None, None, None, None, 4, None, 0, 2, 64, 16, 8, 1, None) == ts.TS_OK
    assert lib.ts_kv_append(vp, vp, vp, vp, vp, 4, vp, 2, 0, 64, 16, 8, 1, None) == ts.TS_ERR_INVALID_ARG
    assert lib.ts_merge_states(None, None, None, None, None, None, 0, 64, 1, None) == ts.TS_OK
    assert lib.ts_merge_states(vp, vp, vp, vp, vp, vp, 3, 12, 1, None) == ts.TS_ERR_UNSUPPORTED
    unaligned = ctypes.c_void_p(24)
    assert lib.ts_merge_states(unaligned, vp, vp, vp, vp, vp, 3, 64, 1, None) == ts.TS_ERR_INVALID_ARG


def test_pool_rows_beyond_int32_are_rejected_before_any_launch(lib):
    """Pools may exceed 4 GiB (64-bit byte offsets), but num_pages * page_size
    rows must stay below 2^31 (32-bit TMA row coordinates): every attention
    entry point rejects more as an argument error, the tensor-core
    multi-query shape included, without touching the device."""
    vp = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    P = (1 << 27)  # x 16 rows = 2^31
    assert lib.ts_paged_decode_attn(vp, vp, vp, vp, 4, vp, 2, 32, 8, 128, 16, P, 1.0, 1, vp, None, vp,
                                    1 << 20, None) == ts.TS_ERR_INVALID_ARG
    assert lib.ts_paged_decode_multi_attn(vp, vp, vp, vp, 4, vp, 2, 4, 32, 8, 128, 16, P, 1.0, 1, vp, None,
                                          vp, 1 << 20, None) == ts.TS_ERR_INVALID_ARG
    groups = ts.PrefixGroupsC()  # zeroed: never read, the size check comes first
    assert lib.ts_cascade_decode_attn(vp, vp, vp, ctypes.byref(groups), vp, 4, vp, 2, 32, 8, 64, 16, P, 1.0, 1,
                                      vp, None, vp, 1 << 20, None) == ts.TS_ERR_INVALID_ARG
    assert lib.ts_mla_paged_decode(vp, vp, vp, 4, vp, 2, 128, 576, 512, 64, (1 << 25), 1.0, vp, None, vp,
                                   1 << 20, None) == ts.TS_ERR_INVALID_ARG


def test_window_and_multi_query_entry_points_validate_before_any_launch(lib):
    """Empty batches are no-ops on every newer entry point; a window below one
    token and a non-finite scale are argument errors; nothing touches a device."""
    vp = ctypes.c_void_p(16)
    # ts_paged_decode_window_attn(q, k, v, bt, bt_stride, lens, B, H_q, H_kv, D, ps, P, window, scale, dt, ...)
    assert lib.ts_paged_decode_window_attn(None, None, None, None, 4, None, 0, 32, 8, 128, 16, 8, 64, 1.0, 1,
                                           None, None, None, 0, None) == ts.TS_OK
    assert lib.ts_paged_decode_window_attn(vp, vp, vp, vp, 4, vp, 2, 32, 8, 128, 16, 8, 0, 1.0, 1,
                                           vp, None, vp, 1 << 20, None) == ts.TS_ERR_INVALID_ARG
    assert b"window" in lib.ts_last_error_detail()
    assert lib.ts_paged_decode_window_attn(vp, vp, vp, vp, 4, vp, 2, 32, 8, 128, 16, 8, 64, float("inf"), 1,
                                           vp, None, vp, 1 << 20, None) == ts.TS_ERR_INVALID_ARG
    # ts_paged_decode_multi_attn: B = 0 with a tensor-core shape, then a non-finite scale
    assert lib.ts_paged_decode_multi_attn(None, None, None, None, 4, None, 0, 4, 32, 8, 128, 16, 8, 1.0, 1,
                                          None, None, None, 0, None) == ts.TS_OK
    assert lib.ts_paged_decode_multi_attn(vp, vp, vp, vp, 4, vp, 2, 4, 32, 8, 128, 16, 8, float("nan"), 1,
                                          vp, None, vp, 1 << 20, None) == ts.TS_ERR_INVALID_ARG
    # ts_paged_decode_fp8_attn: B = 0
    assert lib.ts_paged_decode_fp8_attn(None, None, None, None, None, None, 4, None, 0, 32, 8, 128, 16, 8, 1.0,
                                        None, None, None, 0, None) == ts.TS_OK


def test_python_binding_requires_int32_metadata():
    import torch
    q = torch.zeros(1, 8, 64)
    with pytest.raises(TypeError):
        ts.ts_paged_decode_attn(q, torch.zeros(2, 16, 2, 64), torch.zeros(2, 16, 2, 64),
                                torch.zeros(1, 1, dtype=torch.int64), torch.zeros(1, dtype=torch.int32), 1.0)


def test_launch_trace_toggles_without_a_gpu(lib):
    """Enabling, disabling and collecting the launch trace touches no device
    when nothing was launched: an empty collect returns 0 records."""
    assert lib.ts_trace_enable(1) == ts.TS_OK
    assert lib.ts_trace_enable(0) == ts.TS_OK
    assert lib.ts_trace_collect(None, 0) == 0
    assert ts.ts_trace_collect() == []


def test_fold_sq_factor_host_helper_matches_the_rule(lib):
    """ts_fold_sq_factor is host logic: checked against the oracle's statement
    of the page's rule over a grid, and 0 for non-positive arguments."""
    import oracle
    for H in (1, 4, 16, 48, 64, 100, 128, 200):
        for q_len in range(1, 13):
            for tile in (8, 64, 128):
                assert lib.ts_fold_sq_factor(H, q_len, tile) == oracle.fold_sq_factor(H, q_len, tile)
    assert lib.ts_fold_sq_factor(0, 4, 128) == 0 and lib.ts_fold_sq_factor(64, 0, 128) == 0


def test_binding_constants_match_the_header():
    text = open(os.path.join(ROOT, "include", "ts_attn.h")).read()
    m = re.search(r"#define TS_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", text)
    assert m, "TS_NOALLOC_SCRATCH_BYTES not found"
    assert int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == ts.TS_NOALLOC_SCRATCH_BYTES
    for name in ("TS_DEVERR_PAGE_RANGE", "TS_DEVERR_TIMEOUT", "TS_DEVERR_SMEM_ALIGN"):
        v = re.search(rf"#define {name} (0x[0-9a-fA-F]+|\d+)u?", text) or re.search(rf"\b{name}\s*=\s*(0x[0-9a-fA-F]+|\d+)", text)
        assert v, name
        assert int(v.group(1), 0) == getattr(ts, name), name


def test_clock_stamp_validates_before_any_launch(lib):
    """The measurement aid rejects a null or unaligned buffer and a count out
    of range without enqueueing anything."""
    assert lib.ts_clock_stamp(None, 4, None) == ts.TS_ERR_INVALID_ARG
    assert lib.ts_clock_stamp(ctypes.c_void_p(16), 0, None) == ts.TS_ERR_INVALID_ARG
    assert lib.ts_clock_stamp(ctypes.c_void_p(16), 65536, None) == ts.TS_ERR_INVALID_ARG
    assert lib.ts_clock_stamp(ctypes.c_void_p(20), 4, None) == ts.TS_ERR_INVALID_ARG
