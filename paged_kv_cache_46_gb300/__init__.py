"""Python binding of the ts_attn C library (decode attention over a paged KV cache).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels. Tensors are torch tensors on the current CUDA device; their raw
pointers, sizes and the current stream are passed straight to the C ABI in
``include/ts_attn.h``. Functions keep the C names. Output tensors and
workspaces may be passed in; when omitted they are allocated with torch (the C
library itself never allocates device memory).

The shared library is built in-tree by ``paged_kv_cache_46_gb300.build``.
Importing this package does not need a GPU; calling a kernel does, and there
is no CPU fallback: a missing library raises immediately.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libts_attn.so")

TS_OK, TS_ERR_INVALID_ARG, TS_ERR_UNSUPPORTED, TS_ERR_WORKSPACE, TS_ERR_CUDA, TS_ERR_CAPACITY = range(6)
TS_F32, TS_BF16 = 0, 1
TS_DEVERR_PAGE_RANGE, TS_DEVERR_TIMEOUT, TS_DEVERR_SMEM_ALIGN, TS_DEVERR_TREE = 0x1, 0x2, 0x4, 0x8
TS_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024   # include/ts_attn.h


class TSError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{status_string(status)}: {detail}")
        self.status = status
        self.detail = detail


class PrefixGroupsC(ctypes.Structure):
    _fields_ = [
        ("num_groups", ctypes.c_int32),
        ("prefix_indptr", ctypes.c_void_p),
        ("prefix_pages", ctypes.c_void_p),
        ("prefix_len", ctypes.c_void_p),
        ("member_indptr", ctypes.c_void_p),
        ("member_ids", ctypes.c_void_p),
        ("group_of", ctypes.c_void_p),
        ("capacity_groups", ctypes.c_int32),
        ("capacity_prefix_pages", ctypes.c_int32),
        ("capacity_members", ctypes.c_int32),
    ]


class PrefixForestC(ctypes.Structure):
    _fields_ = [
        ("num_nodes", ctypes.c_int32),
        ("num_levels", ctypes.c_int32),
        ("level_indptr", ctypes.c_void_p),
        ("parent", ctypes.c_void_p),
        ("prefix_indptr", ctypes.c_void_p),
        ("prefix_pages", ctypes.c_void_p),
        ("prefix_len", ctypes.c_void_p),
        ("member_indptr", ctypes.c_void_p),
        ("member_ids", ctypes.c_void_p),
        ("group_of", ctypes.c_void_p),
        ("capacity_nodes", ctypes.c_int32),
        ("capacity_levels", ctypes.c_int32),
        ("capacity_prefix_pages", ctypes.c_int32),
        ("capacity_members", ctypes.c_int32),
    ]


class LaunchRecordC(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_char * 48), ("ms", ctypes.c_float)]


_VP, _I32, _I64, _F32, _SZ, _U32P = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_float, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32))

_SIGNATURES = {
    "ts_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ts_last_error_detail": (ctypes.c_char_p, []),
    "ts_version": (ctypes.c_char_p, []),
    "ts_kv_append": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32, _I32,
                                    ctypes.c_int, _VP]),
    "ts_paged_decode_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "ts_paged_decode_attn": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32, _I32,
                                            _I32, _F32, ctypes.c_int, _VP, _VP, _VP, _SZ, _VP]),
    "ts_paged_decode_attn_noalloc": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32,
                                                    _I32, _I32, _F32, ctypes.c_int, _VP, _VP, _VP]),
    "ts_paged_decode_window_attn": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32, _I32,
                                                   _I32, _I32, _F32, ctypes.c_int, _VP, _VP, _VP, _SZ, _VP]),
    "ts_paged_decode_multi_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "ts_paged_decode_multi_attn": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32, _I32,
                                                  _I32, _I32, _F32, ctypes.c_int, _VP, _VP, _VP, _SZ, _VP]),
    "ts_fold_sq_factor": (_I32, [_I32, _I32, _I32]),
    "ts_kv_append_fp8": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32,
                                        _I32, ctypes.c_int, _VP]),
    "ts_paged_decode_fp8_attn": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32,
                                                _I32, _I32, _F32, _VP, _VP, _VP, _SZ, _VP]),
    "ts_merge_states": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I32, ctypes.c_int, _VP]),
    "ts_group_prefixes": (ctypes.c_int, [_VP, _I32, _VP, _I32, _I32, _I32, ctypes.POINTER(PrefixGroupsC)]),
    "ts_group_prefixes_nested": (ctypes.c_int, [_VP, _I32, _VP, _I32, _I32, _I32, ctypes.POINTER(PrefixForestC)]),
    "ts_cascade_decode_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "ts_cascade_nested_decode_attn": (ctypes.c_int, [_VP, _VP, _VP, ctypes.POINTER(PrefixForestC), _VP, _VP, _I32,
                                                     _VP, _I32, _I32, _I32, _I32, _I32, _I32, _F32, ctypes.c_int,
                                                     _VP, _VP, _VP, _SZ, _VP]),
    "ts_cascade_decode_attn": (ctypes.c_int, [_VP, _VP, _VP, ctypes.POINTER(PrefixGroupsC), _VP, _I32, _VP,
                                              _I32, _I32, _I32, _I32, _I32, _I32, _F32, ctypes.c_int,
                                              _VP, _VP, _VP, _SZ, _VP]),
    "ts_mla_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "ts_mla_paged_decode": (ctypes.c_int, [_VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32, _I32, _I32,
                                           _F32, _VP, _VP, _VP, _SZ, _VP]),
    "ts_mla_multi_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "ts_mla_paged_decode_multi": (ctypes.c_int, [_VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32, _I32, _I32,
                                                 _I32, _F32, _VP, _VP, _VP, _SZ, _VP]),
    "ts_paged_decode_tree_attn": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _VP, _VP, _I32, _I32, _I32, _I32, _I32,
                                                 _I32, _I32, _F32, _I32, _VP, _VP, _VP, _SZ, _VP]),
    "ts_mla_paged_decode_fp8": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _I32, _I32, _I32, _I32,
                                               _I32, _I32, _F32, _VP, _VP, _VP, _SZ, _VP]),
    "ts_read_device_error": (ctypes.c_int, [_VP, _U32P, _VP]),
    "ts_trace_enable": (ctypes.c_int, [_I32]),
    "ts_trace_collect": (_I32, [ctypes.POINTER(LaunchRecordC), _I32]),
    "ts_clock_stamp": (ctypes.c_int, [_VP, _I32, _VP]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m paged_kv_cache_46_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().ts_status_string(int(status)).decode()
    except Exception:  # library not loadable: still describe the code
        return {0: "TS_OK"}.get(int(status), f"status {status}")


def _check(status: int):
    if status != TS_OK:
        raise TSError(status, lib().ts_last_error_detail().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TS_F32
    if t.dtype == torch.bfloat16:
        return TS_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _require_i32(*ts):
    for t in ts:
        if t.dtype != torch.int32:
            raise TypeError("block tables, lengths and positions must be int32")


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def ts_kv_append(k_new, v_new, k_pool, v_pool, block_table, positions, stream=None) -> None:
    """Write k_new/v_new [B, H_kv, D] into the pools at ``positions`` (see ts_attn.h)."""
    _require_i32(block_table, positions)
    B, H_kv, D = k_new.shape
    _check(lib().ts_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                              block_table.shape[1], _ptr(positions), B, H_kv, D, k_pool.shape[1],
                              k_pool.shape[0], _dt(k_pool), _stream(stream)))


def ts_paged_decode_workspace_size(B: int, H_q: int, D: int) -> int:
    return int(lib().ts_paged_decode_workspace_size(B, H_q, D))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed, 256-byte aligned uint8 workspace (torch's allocator aligns to >= 256)."""
    ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")
    assert ws.data_ptr() % 256 == 0
    return ws


def ts_paged_decode_attn(q, k_pool, v_pool, block_table, seq_lens, scale: float, out=None, lse=None,
                         workspace=None, stream=None, return_lse: bool = False):
    """Decode attention over a paged cache; returns ``out`` (and ``lse``)."""
    _require_i32(block_table, seq_lens)
    B, H_q, D = q.shape
    P, ps, H_kv, _ = k_pool.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, H_q, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(ts_paged_decode_workspace_size(B, H_q, D), q.device)
    _check(lib().ts_paged_decode_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                      block_table.shape[1], _ptr(seq_lens), B, H_q, H_kv, D, ps, P,
                                      float(scale), _dt(q), _ptr(out), _ptr(lse), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)))
    return (out, lse) if return_lse else out


def ts_paged_decode_window_attn(q, k_pool, v_pool, block_table, seq_lens, scale: float, window: int, out=None,
                                lse=None, workspace=None, stream=None, return_lse: bool = False):
    """Decode attention over a sliding-window KV group (each query attends its
    sequence's last ``window`` tokens); returns ``out`` (and ``lse``)."""
    _require_i32(block_table, seq_lens)
    B, H_q, D = q.shape
    P, ps, H_kv, _ = k_pool.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, H_q, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(ts_paged_decode_workspace_size(B, H_q, D), q.device)
    _check(lib().ts_paged_decode_window_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                             block_table.shape[1], _ptr(seq_lens), B, H_q, H_kv, D, ps, P,
                                             int(window), float(scale), _dt(q), _ptr(out), _ptr(lse),
                                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                                             _stream(stream)))
    return (out, lse) if return_lse else out


def ts_paged_decode_attn_noalloc(q, k_pool, v_pool, block_table, seq_lens, scale: float, out, lse=None,
                                 stream=None) -> None:
    """ts_paged_decode_attn for callers that cannot allocate device memory.

    The library takes its split-KV scratch from a fixed array in its own device
    image (TS_NOALLOC_SCRATCH_BYTES, one per GPU, kept until exit) instead of a
    caller workspace. ``out`` (and ``lse`` if wanted) must be passed in: this
    wrapper allocates nothing either. Calls that may overlap on one GPU share
    the array and race; see include/ts_attn.h.
    """
    _require_i32(block_table, seq_lens)
    B, H_q, D = q.shape
    P, ps, H_kv, _ = k_pool.shape
    _check(lib().ts_paged_decode_attn_noalloc(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                              block_table.shape[1], _ptr(seq_lens), B, H_q, H_kv, D, ps, P,
                                              float(scale), _dt(q), _ptr(out), _ptr(lse), _stream(stream)))


def ts_paged_decode_multi_workspace_size(B: int, q_len: int, H_q: int, D: int) -> int:
    return int(lib().ts_paged_decode_multi_workspace_size(B, q_len, H_q, D))


def ts_fold_sq_factor(num_heads: int, q_len: int, tile_rows: int = 128) -> int:
    """Query tokens folded into a tile's rows (see include/ts_attn.h)."""
    return int(lib().ts_fold_sq_factor(num_heads, q_len, tile_rows))


def ts_paged_decode_multi_attn(q, k_pool, v_pool, block_table, seq_lens, scale: float, out=None, lse=None,
                               workspace=None, stream=None, return_lse: bool = False):
    """Decode with q_len query tokens per sequence, q [B, q_len, H_q, D]; seq_lens count
    the new tokens (already appended). Returns ``out`` [B, q_len, H_q, D] (and ``lse``)."""
    _require_i32(block_table, seq_lens)
    B, q_len, H_q, D = q.shape
    P, ps, H_kv, _ = k_pool.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, q_len, H_q, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(ts_paged_decode_multi_workspace_size(B, q_len, H_q, D), q.device)
    _check(lib().ts_paged_decode_multi_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                            block_table.shape[1], _ptr(seq_lens), B, q_len, H_q, H_kv, D,
                                            ps, P, float(scale), _dt(q), _ptr(out), _ptr(lse),
                                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                                            _stream(stream)))
    return (out, lse) if return_lse else out


def _require_fp8_cache(k_pool, v_pool, k_scale, v_scale):
    if k_pool.dtype != torch.uint8 or v_pool.dtype != torch.uint8:
        raise TypeError("fp8 pools hold e4m3fn codes as uint8")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32:
        raise TypeError("fp8 scales are float32 [num_pages, page_size, H_kv]")
    if tuple(k_scale.shape) != tuple(k_pool.shape[:3]) or tuple(v_scale.shape) != tuple(v_pool.shape[:3]):
        raise ValueError("scales must be [num_pages, page_size, H_kv] of their pool")


def ts_kv_append_fp8(k_new, v_new, k_pool, v_pool, k_scale, v_scale, block_table, positions,
                     stream=None) -> None:
    """Quantize k_new/v_new [B, H_kv, D] into fp8 pools and their scales (see ts_attn.h)."""
    _require_i32(block_table, positions)
    _require_fp8_cache(k_pool, v_pool, k_scale, v_scale)
    B, H_kv, D = k_new.shape
    _check(lib().ts_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
                                  _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(positions), B,
                                  H_kv, D, k_pool.shape[1], k_pool.shape[0], _dt(k_new), _stream(stream)))


def ts_paged_decode_fp8_attn(q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, scale: float,
                             out=None, lse=None, workspace=None, stream=None, return_lse: bool = False):
    """Decode attention over an fp8 (e4m3fn) cache with bf16 queries; returns ``out`` (and ``lse``)."""
    _require_i32(block_table, seq_lens)
    _require_fp8_cache(k_pool, v_pool, k_scale, v_scale)
    B, H_q, D = q.shape
    P, ps, H_kv, _ = k_pool.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, H_q, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(ts_paged_decode_workspace_size(B, H_q, D), q.device)
    _check(lib().ts_paged_decode_fp8_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
                                          _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H_q, H_kv,
                                          D, ps, P, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))
    return (out, lse) if return_lse else out


def ts_merge_states(o_a, lse_a, o_b, lse_b, o_out=None, lse_out=None, stream=None):
    """LSE-merge two states [rows, D] (+ [rows] LSE); returns (o_out, lse_out)."""
    D = o_a.shape[-1]
    rows = o_a.numel() // D
    if o_out is None:
        o_out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    _check(lib().ts_merge_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out), _ptr(lse_out),
                                 rows, D, _dt(o_a), _stream(stream)))
    return o_out, lse_out


def ts_group_prefixes(block_table: np.ndarray, seq_lens: np.ndarray, page_size: int, min_group: int = 2):
    """Host greedy longest-shared-prefix grouping; returns a dict of int32 numpy arrays."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = lens.shape[0]
    cap_g = max(1, B // max(2, min_group))
    caps = np.maximum(0, (lens.astype(np.int64) - 1) // page_size)
    cap_pages = max(1, int(min(int(caps.sum()), cap_g * bt.shape[1])))
    # the library writes every entry it reports; nothing needs clearing
    arrays = {
        "prefix_indptr": np.empty(cap_g + 1, np.int32), "prefix_pages": np.empty(cap_pages, np.int32),
        "prefix_len": np.empty(cap_g, np.int32), "member_indptr": np.empty(cap_g + 1, np.int32),
        "member_ids": np.empty(max(1, B), np.int32), "group_of": np.empty(max(1, B), np.int32),
    }
    c = PrefixGroupsC(0, *[arrays[k].ctypes.data for k in
                           ("prefix_indptr", "prefix_pages", "prefix_len", "member_indptr", "member_ids",
                            "group_of")], cap_g, cap_pages, max(1, B))
    _check(lib().ts_group_prefixes(bt.ctypes.data, bt.shape[1], lens.ctypes.data, B, page_size, min_group,
                                   ctypes.byref(c)))
    G = c.num_groups
    return {
        "num_groups": G,
        "prefix_indptr": arrays["prefix_indptr"][:G + 1].copy(),
        "prefix_pages": arrays["prefix_pages"][:arrays["prefix_indptr"][G]].copy(),
        "prefix_len": arrays["prefix_len"][:G].copy(),
        "member_indptr": arrays["member_indptr"][:G + 1].copy(),
        "member_ids": arrays["member_ids"][:arrays["member_indptr"][G]].copy(),
        "group_of": arrays["group_of"][:B].copy(),
    }


def ts_group_prefixes_nested(block_table: np.ndarray, seq_lens: np.ndarray, page_size: int,
                             min_group: int = 2):
    """Host greedy shared-prefix search kept as a tree; returns a dict of int32 numpy arrays
    (nodes level by level, see ts_prefix_forest in ts_attn.h)."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = lens.shape[0]
    caps = np.maximum(0, (lens.astype(np.int64) - 1) // page_size)
    cap_n = max(1, B)               # every node has >= 2 members and its own sequence set
    cap_l = max(1, int(caps.max()) if B else 1)
    cap_pages = max(1, int(caps.sum()))
    cap_members = max(1, int(caps.sum()))  # a sequence is in at most one node per shared page
    while True:
        arrays = {
            "level_indptr": np.empty(cap_l + 1, np.int32), "parent": np.empty(cap_n, np.int32),
            "prefix_indptr": np.empty(cap_n + 1, np.int32), "prefix_pages": np.empty(cap_pages, np.int32),
            "prefix_len": np.empty(cap_n, np.int32), "member_indptr": np.empty(cap_n + 1, np.int32),
            "member_ids": np.empty(cap_members, np.int32), "group_of": np.empty(max(1, B), np.int32),
        }
        c = PrefixForestC(0, 0, *[arrays[k].ctypes.data for k in
                                  ("level_indptr", "parent", "prefix_indptr", "prefix_pages", "prefix_len",
                                   "member_indptr", "member_ids", "group_of")],
                          cap_n, cap_l, cap_pages, cap_members)
        st = lib().ts_group_prefixes_nested(bt.ctypes.data, bt.shape[1], lens.ctypes.data, B, page_size,
                                            min_group, ctypes.byref(c))
        if st != TS_ERR_CAPACITY:
            break
        cap_n, cap_l = max(cap_n, c.num_nodes), max(cap_l, c.num_levels)
        cap_members *= 2
    _check(st)
    N, L = c.num_nodes, c.num_levels
    return {
        "num_nodes": N, "num_levels": L,
        "level_indptr": arrays["level_indptr"][:L + 1].copy() if N else np.zeros(1, np.int32),
        "parent": arrays["parent"][:N].copy(),
        "prefix_indptr": arrays["prefix_indptr"][:N + 1].copy(),
        "prefix_pages": arrays["prefix_pages"][:arrays["prefix_indptr"][N]].copy(),
        "prefix_len": arrays["prefix_len"][:N].copy(),
        "member_indptr": arrays["member_indptr"][:N + 1].copy(),
        "member_ids": arrays["member_ids"][:arrays["member_indptr"][N]].copy(),
        "group_of": arrays["group_of"][:B].copy(),
    }


def forest_to_device(forest: dict, device="cuda") -> dict:
    """Device int32 copies of the arrays of ts_group_prefixes_nested (plus the host level_indptr)."""
    out = {"num_nodes": int(forest["num_nodes"]), "num_levels": int(forest["num_levels"]),
           "level_indptr_host": np.ascontiguousarray(forest["level_indptr"], dtype=np.int32)}
    for k in ("level_indptr", "parent", "prefix_indptr", "prefix_pages", "prefix_len", "member_indptr",
              "member_ids", "group_of"):
        a = forest[k] if len(forest[k]) else np.zeros(1, np.int32)
        out[k] = torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    return out


def ts_cascade_nested_decode_attn(q, k_pool, v_pool, forest_dev: dict, block_table, seq_lens, scale: float,
                                  out=None, lse=None, workspace=None, stream=None, return_lse: bool = False):
    """Cascade decode over a nested prefix forest (device arrays from forest_to_device)."""
    _require_i32(block_table, seq_lens)
    B, H_q, D = q.shape
    P, ps, H_kv, _ = k_pool.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, H_q, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(ts_cascade_decode_workspace_size(B, H_q, D), q.device)
    f = forest_dev
    c = PrefixForestC(f["num_nodes"], f["num_levels"], *[f[k].data_ptr() for k in
                                                         ("level_indptr", "parent", "prefix_indptr", "prefix_pages",
                                                          "prefix_len", "member_indptr", "member_ids", "group_of")],
                      0, 0, 0, 0)
    lvl = f["level_indptr_host"]
    _check(lib().ts_cascade_nested_decode_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), ctypes.byref(c),
                                               lvl.ctypes.data, _ptr(block_table), block_table.shape[1],
                                               _ptr(seq_lens), B, H_q, H_kv, D, ps, P, float(scale), _dt(q),
                                               _ptr(out), _ptr(lse), _ptr(workspace),
                                               workspace.numel() * workspace.element_size(), _stream(stream)))
    return (out, lse) if return_lse else out


def groups_to_device(groups: dict, device="cuda") -> dict:
    """Device int32 copies of the CSR arrays of ts_group_prefixes."""
    out = {"num_groups": int(groups["num_groups"])}
    for k in ("prefix_indptr", "prefix_pages", "prefix_len", "member_indptr", "member_ids", "group_of"):
        a = groups[k] if len(groups[k]) else np.zeros(1, np.int32)
        out[k] = torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    return out


def ts_cascade_decode_workspace_size(B: int, H_q: int, D: int) -> int:
    return int(lib().ts_cascade_decode_workspace_size(B, H_q, D))


def ts_cascade_decode_attn(q, k_pool, v_pool, groups_dev: dict, block_table, seq_lens, scale: float,
                           out=None, lse=None, workspace=None, stream=None, return_lse: bool = False):
    """Shared-prefix (cascade) decode attention; ``groups_dev`` from :func:`groups_to_device`."""
    _require_i32(block_table, seq_lens)
    B, H_q, D = q.shape
    P, ps, H_kv, _ = k_pool.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, H_q, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(ts_cascade_decode_workspace_size(B, H_q, D), q.device)
    g = groups_dev
    c = PrefixGroupsC(g["num_groups"], _ptr(g["prefix_indptr"]), _ptr(g["prefix_pages"]), _ptr(g["prefix_len"]),
                      _ptr(g["member_indptr"]), _ptr(g["member_ids"]), _ptr(g["group_of"]), 0, 0, 0)
    _check(lib().ts_cascade_decode_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), ctypes.byref(c), _ptr(block_table),
                                        block_table.shape[1], _ptr(seq_lens), B, H_q, H_kv, D, ps, P,
                                        float(scale), _dt(q), _ptr(out), _ptr(lse), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)))
    return (out, lse) if return_lse else out


def ts_mla_workspace_size(B: int, H: int, D_v: int) -> int:
    return int(lib().ts_mla_workspace_size(B, H, D_v))


def ts_mla_paged_decode(q, kv_pool, block_table, seq_lens, scale: float, d_v: int = 512, out=None, lse=None,
                        workspace=None, stream=None, return_lse: bool = False):
    """Absorbed-MLA decode: q [B, H, Dqk] bf16, kv_pool [P, ps, Dqk] bf16 -> out [B, H, d_v]."""
    _require_i32(block_table, seq_lens)
    B, H, Dqk = q.shape
    P, ps, _ = kv_pool.shape
    if out is None:
        out = torch.empty(B, H, d_v, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(B, H, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(ts_mla_workspace_size(B, H, d_v), q.device)
    _check(lib().ts_mla_paged_decode(_ptr(q), _ptr(kv_pool), _ptr(block_table), block_table.shape[1],
                                     _ptr(seq_lens), B, H, Dqk, d_v, ps, P, float(scale), _ptr(out), _ptr(lse),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))
    return (out, lse) if return_lse else out


def ts_paged_decode_tree_attn(q, k_pool, v_pool, block_table, seq_lens, parents, scale: float, out=None,
                              lse=None, workspace=None, stream=None, return_lse: bool = False):
    """Tree verification: q [B, n, H_q, D] bf16, parents int32 [B, n] (-1 or an
    earlier draft token) -> out [B, n, H_q, D]."""
    _require_i32(block_table, seq_lens, parents)
    B, n, H_q, D = q.shape
    P, ps, H_kv, _ = k_pool.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, n, H_q, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(256, q.device)
    _check(lib().ts_paged_decode_tree_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                           block_table.shape[1], _ptr(seq_lens), _ptr(parents), B, n, H_q, H_kv, D,
                                           ps, P, float(scale), _dt(q), _ptr(out), _ptr(lse), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream)))
    return (out, lse) if return_lse else out


def ts_mla_multi_workspace_size(B: int, q_len: int, H: int, D_v: int) -> int:
    return int(lib().ts_mla_multi_workspace_size(B, q_len, H, D_v))


def ts_mla_paged_decode_multi(q, kv_pool, block_table, seq_lens, scale: float, d_v: int = 512, out=None,
                              lse=None, workspace=None, stream=None, return_lse: bool = False):
    """Absorbed-MLA decode of q_len tokens per sequence: q [B, q_len, H, Dqk] bf16,
    kv_pool [P, ps, Dqk] bf16 -> out [B, q_len, H, d_v]."""
    _require_i32(block_table, seq_lens)
    B, q_len, H, Dqk = q.shape
    P, ps, _ = kv_pool.shape
    if out is None:
        out = torch.empty(B, q_len, H, d_v, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(B, q_len, H, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(ts_mla_multi_workspace_size(B, q_len, H, d_v), q.device)
    _check(lib().ts_mla_paged_decode_multi(_ptr(q), _ptr(kv_pool), _ptr(block_table), block_table.shape[1],
                                           _ptr(seq_lens), B, q_len, H, Dqk, d_v, ps, P, float(scale), _ptr(out),
                                           _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)))
    return (out, lse) if return_lse else out


def ts_mla_paged_decode_fp8(q_codes, q_scale, kv_codes, kv_scale, block_table, seq_lens, scale: float,
                            d_v: int = 512, out=None, lse=None, workspace=None, stream=None, return_lse: bool = False):
    """Absorbed-MLA decode on e4m3 inputs: q_codes uint8 [B, H, 576] or [B, q_len, H, 576]
    with q_scale float32 [B, (q_len,) H]; kv_codes uint8 [P, ps, 576] with kv_scale
    float32 [P, ps] -> out bf16 [B, (q_len,) H, d_v]."""
    _require_i32(block_table, seq_lens)
    if q_codes.dtype != torch.uint8 or kv_codes.dtype != torch.uint8:
        raise TypeError("fp8 codes travel as uint8 tensors")
    if q_scale.dtype != torch.float32 or kv_scale.dtype != torch.float32:
        raise TypeError("scales must be float32")
    single = q_codes.dim() == 3
    B, q_len, H, Dqk = (q_codes.shape[0], 1, *q_codes.shape[1:]) if single else q_codes.shape
    P, ps, _ = kv_codes.shape
    shape = (B, H) if single else (B, q_len, H)
    if out is None:
        out = torch.empty(*shape, d_v, dtype=torch.bfloat16, device=q_codes.device)
    if lse is None and return_lse:
        lse = torch.empty(*shape, dtype=torch.float32, device=q_codes.device)
    if workspace is None:
        workspace = new_workspace(ts_mla_multi_workspace_size(B, q_len, H, d_v), q_codes.device)
    _check(lib().ts_mla_paged_decode_fp8(_ptr(q_codes), _ptr(q_scale), _ptr(kv_codes), _ptr(kv_scale),
                                         _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, q_len, H, Dqk,
                                         d_v, ps, P, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream)))
    return (out, lse) if return_lse else out


def ts_read_device_error(workspace, stream=None) -> int:
    """Sticky device error bits of a workspace; None reads those of the
    allocation-free entry point's static scratch on the current device."""
    v = ctypes.c_uint32(0)
    _check(lib().ts_read_device_error(_ptr(workspace), ctypes.byref(v), _stream(stream)))
    return int(v.value)


def ts_trace_enable(on: bool) -> None:
    _check(lib().ts_trace_enable(1 if on else 0))


def ts_clock_stamp(stamps, stream=None) -> None:
    """Enqueues one clock stamp per row of ``stamps`` (an int64 device tensor
    [n, 3]): SM id, that SM's cycle counter, global timer in ns."""
    if stamps.dtype != torch.int64 or stamps.dim() != 2 or stamps.shape[1] != 3 or not stamps.is_contiguous():
        raise TSError(TS_ERR_INVALID_ARG, "ts_clock_stamp: stamps must be a contiguous int64 tensor [n, 3]")
    _check(lib().ts_clock_stamp(_ptr(stamps), stamps.shape[0], _stream(stream)))


def ts_trace_collect(capacity: int = 4096):
    """[(kernel name, device ms)] of the launches recorded since the last collect."""
    buf = (LaunchRecordC * capacity)()
    n = lib().ts_trace_collect(buf, capacity)
    if n < 0:
        raise TSError(TS_ERR_CUDA, lib().ts_last_error_detail().decode())
    return [(buf[i].kernel.decode(), float(buf[i].ms)) for i in range(min(n, capacity))]
