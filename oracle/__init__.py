"""Plain CPU oracle for batched variable-length exact top-K.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.
The product library never loads it and shares no code with it.

The arithmetic lives in ``topk_oracle.c`` (plain C, fp64 comparisons,
``qsort`` by value descending then column ascending); this module only
compiles it with the host C compiler and marshals arrays through ctypes.
Every function cites the passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

DTYPE_CODES = {"float32": 0, "bfloat16": 1, "float16": 2}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, -O2, no -march)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.oracle_row_length.restype = i64
            lib.oracle_row_length.argtypes = [i64, i64, i64, i64, i64]
            lib.oracle_ragged_length.restype = i64
            lib.oracle_ragged_length.argtypes = [i64, i64, i64]
            lib.oracle_select_row.restype = ctypes.c_int
            lib.oracle_select_row.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp]
            lib.oracle_topk_varlen.restype = ctypes.c_int
            lib.oracle_topk_varlen.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp,
                                               i32, i32, i32, vp, vp]
            lib.oracle_page_table_transform.restype = ctypes.c_int
            lib.oracle_page_table_transform.argtypes = [
                vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, i64, i64, vp, i32, i32,
                vp, vp]
            lib.oracle_topk_varlen_ties.restype = ctypes.c_int
            lib.oracle_topk_varlen_ties.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp,
                                                    i32, i32, i32, ctypes.c_int, vp, vp]
            lib.oracle_select_row_large_ties.restype = ctypes.c_int
            lib.oracle_select_row_large_ties.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp]
            lib.oracle_ragged_offset_transform.restype = ctypes.c_int
            lib.oracle_ragged_offset_transform.argtypes = [
                vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, i32, vp]
            lib.oracle_seqs_page_table_transform.restype = ctypes.c_int
            lib.oracle_seqs_page_table_transform.argtypes = [
                vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, i64, i64, vp, i64, i32, vp]
            _lib = lib
    return _lib


def _dtype_name(t) -> str:
    return str(t.dtype).replace("torch.", "")


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return a.data_ptr()


def row_length(seq_len: int, next_n: int, t: int, compress_ratio: int, width: int) -> int:
    """Valid columns of row t of a request (FlashInfer `top_k_varlen`, `seq_lens`)."""
    return int(_load().oracle_row_length(seq_len, next_n, t, compress_ratio, width))


def row_lengths(seq_lens, num_rows: int, next_n: int, compress_ratio: int, width: int):
    """Per-row valid column counts for a whole batch, as an int64 numpy array."""
    sl = np.asarray(seq_lens, dtype=np.int64)
    lib = _load()
    return np.array([lib.oracle_row_length(int(sl[r // next_n]), next_n, r % next_n,
                                           compress_ratio, width)
                     for r in range(num_rows)], dtype=np.int64)


def ragged_length(length: int, row_start: int, width: int) -> int:
    """Valid columns of a page-table row ([row_start, row_start+len) in width)."""
    return int(_load().oracle_ragged_length(length, row_start, width))


def select_row(row, n: int, k: int, return_values: bool = True):
    """Top-k of the first n entries of a 1-D CPU tensor, (value desc, index asc)."""
    import torch
    row = row.contiguous()
    idx = torch.empty(k, dtype=torch.int32)
    val = torch.empty(k, dtype=row.dtype) if return_values else None
    rc = _load().oracle_select_row(_ptr(row), DTYPE_CODES[_dtype_name(row)], n, k,
                                   _ptr(idx), _ptr(val))
    if rc != 0:
        raise ValueError(f"oracle_select_row failed: {rc}")
    return idx, val


def topk_varlen(logits, seq_lens, top_k: int, next_n: int = 1, compress_ratio: int = 1,
                return_values: bool = True):
    """Oracle of `top_k_varlen` on CPU tensors; returns (indices, values|None).

    ``logits`` may be a row-strided view (inner stride 1)."""
    import torch
    assert logits.dim() == 2 and logits.stride(1) == 1 and logits.device.type == "cpu"
    R, W = logits.shape
    S = logits.stride(0) if R > 1 else W
    sl = seq_lens.to(torch.int32).contiguous()
    idx = torch.empty((R, top_k), dtype=torch.int32)
    val = torch.empty((R, top_k), dtype=logits.dtype) if return_values else None
    rc = _load().oracle_topk_varlen(_ptr(logits), DTYPE_CODES[_dtype_name(logits)], R, W, S,
                                    _ptr(sl), next_n, compress_ratio, top_k, _ptr(idx),
                                    _ptr(val))
    if rc != 0:
        raise ValueError(f"oracle_topk_varlen failed: {rc}")
    return idx, val


def topk_varlen_ties(logits, seq_lens, top_k: int, tie_large: bool, next_n: int = 1,
                     compress_ratio: int = 1, return_values: bool = True):
    """Oracle of `top_k_varlen` with a tie mode (SMALL: smallest columns among
    the values equal to the k-th; LARGE: largest), canonical output order."""
    import torch
    assert logits.dim() == 2 and logits.stride(1) == 1 and logits.device.type == "cpu"
    R, W = logits.shape
    S = logits.stride(0) if R > 1 else W
    sl = seq_lens.to(torch.int32).contiguous()
    idx = torch.empty((R, top_k), dtype=torch.int32)
    val = torch.empty((R, top_k), dtype=logits.dtype) if return_values else None
    rc = _load().oracle_topk_varlen_ties(_ptr(logits), DTYPE_CODES[_dtype_name(logits)], R, W, S,
                                         _ptr(sl), next_n, compress_ratio, top_k,
                                         1 if tie_large else 0, _ptr(idx), _ptr(val))
    if rc != 0:
        raise ValueError(f"oracle_topk_varlen_ties failed: {rc}")
    return idx, val


def page_table_transform(scores, lengths, page_table, top_k: int, page_size: int = 1,
                         row_starts=None, page_table_row_starts=None):
    """Oracle of the fused compact page-table transform; returns (out, out_raw)."""
    import torch
    assert scores.dim() == 2 and scores.stride(1) == 1
    assert page_table.dim() == 2 and page_table.stride(1) == 1
    R, W = scores.shape
    S = scores.stride(0) if R > 1 else W
    ln = lengths.to(torch.int32).contiguous()
    rs = row_starts.to(torch.int32).contiguous() if row_starts is not None else None
    prs = (page_table_row_starts.to(torch.int32).contiguous()
           if page_table_row_starts is not None else None)
    P = page_table.shape[1]
    PS = page_table.stride(0) if page_table.shape[0] > 1 else P
    out = torch.empty((R, top_k), dtype=torch.int32)
    out_raw = torch.empty((R, top_k), dtype=torch.int32)
    rc = _load().oracle_page_table_transform(
        _ptr(scores), DTYPE_CODES[_dtype_name(scores)], R, W, S, _ptr(ln), _ptr(rs),
        _ptr(page_table), P, PS, _ptr(prs), page_size, top_k, _ptr(out), _ptr(out_raw))
    if rc != 0:
        raise ValueError(f"oracle_page_table_transform failed: {rc}")
    return out, out_raw


def ragged_offset_transform(scores, lengths, offsets, top_k: int, row_starts=None):
    """Oracle of the ragged KV offset transform: out = idx + offsets[row]."""
    import torch
    assert scores.dim() == 2 and scores.stride(1) == 1
    R, W = scores.shape
    S = scores.stride(0) if R > 1 else W
    ln = lengths.to(torch.int32).contiguous()
    rs = row_starts.to(torch.int32).contiguous() if row_starts is not None else None
    off = offsets.to(torch.int32).contiguous()
    out = torch.empty((R, top_k), dtype=torch.int32)
    rc = _load().oracle_ragged_offset_transform(
        _ptr(scores), DTYPE_CODES[_dtype_name(scores)], R, W, S, _ptr(ln), _ptr(rs), _ptr(off),
        top_k, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_ragged_offset_transform failed: {rc}")
    return out


def seqs_page_table_transform(scores, lengths, page_table, cu_seqlens_q, top_k: int,
                              row_starts=None):
    """Oracle of the page_size-1 page-table transform over requests
    (row r belongs to request b with cu_seqlens_q[b] <= r < cu_seqlens_q[b+1])."""
    import torch
    assert scores.dim() == 2 and scores.stride(1) == 1
    assert page_table.dim() == 2 and page_table.stride(1) == 1
    R, W = scores.shape
    S = scores.stride(0) if R > 1 else W
    ln = lengths.to(torch.int32).contiguous()
    rs = row_starts.to(torch.int32).contiguous() if row_starts is not None else None
    cu = cu_seqlens_q.to(torch.int32).contiguous()
    P = page_table.shape[1]
    PS = page_table.stride(0) if page_table.shape[0] > 1 else P
    out = torch.empty((R, top_k), dtype=torch.int32)
    rc = _load().oracle_seqs_page_table_transform(
        _ptr(scores), DTYPE_CODES[_dtype_name(scores)], R, W, S, _ptr(ln), _ptr(rs),
        _ptr(page_table), P, PS, _ptr(cu), cu.numel() - 1, top_k, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_seqs_page_table_transform failed: {rc}")
    return out
