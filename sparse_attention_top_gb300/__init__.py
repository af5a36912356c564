"""Batched variable-length exact top-K for the DSA indexer, on GB300.

Thin ctypes binding over the C ABI of ``libgbtopk.so`` (``include/gbtopk.h``).
PyTorch is used only for device memory, streams and pointers: every step of
the selection runs in the library's CUDA kernels.  There is no CPU path; if
the library has not been built the calls raise ``RuntimeError``.

Low-level entry points keep the C names (``gbtopk_varlen``,
``gbtopk_page_table_transform``, ``gbtopk_workspace_bytes``,
``gbtopk_device_status``, ``gbtopk_plan_query``, ``gbtopk_status_str``);
``top_k_varlen`` and ``top_k_page_table_transform`` follow the Python
signatures of the FlashInfer ``top_k_varlen`` page and of the compact
page-table API quoted on the SGLang PR #33237 page.
"""
from __future__ import annotations

import ctypes
import os
import threading
import warnings
from typing import Optional, Tuple

import torch

__all__ = [
    "top_k_varlen", "top_k_page_table_transform", "gbtopk_varlen",
    "gbtopk_page_table_transform", "gbtopk_workspace_bytes", "gbtopk_device_status",
    "gbtopk_plan_query", "gbtopk_status_str", "gbtopk_varlen_static_ws", "library_path",
    "load_library", "top_k_ragged_transform", "top_k_page_table_transform_cu_seqlens",
    "gbtopk_ragged_transform", "gbtopk_page_table_transform_cu_seqlens",
    "GbtopkError", "MAX_TOP_K", "SORTED", "TIE_SMALL", "TIE_LARGE", "order_flags",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libgbtopk.so")
_lib = None
_lock = threading.Lock()

OK, HINT_DISCARDED = 0, 1
EINVAL, EALIGN, EOVERLAP, EUNSUPPORTED, ECUDA, EWORKSPACE, ETIMEOUT = -1, -2, -3, -4, -5, -6, -7
MAX_TOP_K = 16384
# Flags of the C entry points' `deterministic` argument (include/gbtopk.h).
SORTED, TIE_SMALL, TIE_LARGE = 1, 2, 4


def order_flags(deterministic: bool = False, tie_mode: Optional[str] = None) -> int:
    """Flags for ``deterministic`` and a tie mode among values equal to the
    k-th: None (arbitrary, or the smallest columns when ``deterministic``),
    "small" (smallest columns) or "large" (largest columns)."""
    ties = {None: 0, "small": TIE_SMALL, "large": TIE_LARGE}
    if tie_mode not in ties:
        raise ValueError('tie_mode must be None, "small" or "large"')
    return (SORTED if deterministic else 0) | ties[tie_mode]
_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


class GbtopkError(ValueError):
    """A negative status from the library (nothing was enqueued)."""

    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads ``libgbtopk.so`` once; raises if it was never built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"gbtopk CUDA library not found at {_LIB_PATH}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (there is no CPU fallback)")
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
        c_int = ctypes.c_int
        lib.gbtopk_varlen.restype = c_int
        lib.gbtopk_varlen.argtypes = [vp, c_int, i64, i64, i64, vp, i32, i32, i32, vp, vp, vp,
                                      c_int, vp, sz, vp]
        lib.gbtopk_page_table_transform.restype = c_int
        lib.gbtopk_page_table_transform.argtypes = [vp, c_int, i64, i64, i64, vp, vp, vp, i64,
                                                    i64, vp, i32, i32, vp, vp, c_int, vp, sz, vp]
        lib.gbtopk_workspace_bytes.restype = sz
        lib.gbtopk_workspace_bytes.argtypes = [i64, i64, i32, c_int]
        lib.gbtopk_device_status.restype = c_int
        lib.gbtopk_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        lib.gbtopk_plan_query.restype = c_int
        lib.gbtopk_plan_query.argtypes = [i64, i64, i32, c_int, ctypes.POINTER(ctypes.c_int64)]
        lib.gbtopk_varlen_static_ws.restype = c_int
        lib.gbtopk_varlen_static_ws.argtypes = [vp, c_int, i64, i64, i64, vp, i32, i32, i32, vp, vp,
                                                vp, c_int, vp]
        lib.gbtopk_ragged_transform.restype = c_int
        lib.gbtopk_ragged_transform.argtypes = [vp, c_int, i64, i64, i64, vp, vp, vp, i32, vp,
                                                c_int, vp, sz, vp]
        lib.gbtopk_page_table_transform_cu_seqlens.restype = c_int
        lib.gbtopk_page_table_transform_cu_seqlens.argtypes = [
            vp, c_int, i64, i64, i64, vp, vp, vp, i64, i64, vp, i64, i32, vp, c_int, vp, sz, vp]
        lib.gbtopk_status_str.restype = ctypes.c_char_p
        lib.gbtopk_status_str.argtypes = [c_int]
        _lib = lib
        return lib


def gbtopk_status_str(status: int) -> str:
    return load_library().gbtopk_status_str(status).decode()


def _check(status: int) -> int:
    if status < 0:
        raise GbtopkError(status, gbtopk_status_str(status))
    return status


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream_handle(device: torch.device):
    return torch.cuda.current_stream(device).cuda_stream


def gbtopk_workspace_bytes(num_rows: int, width: int, top_k: int, dtype: torch.dtype) -> int:
    return int(load_library().gbtopk_workspace_bytes(num_rows, width, top_k, _DTYPES[dtype]))


def gbtopk_plan_query(num_rows: int, width: int, top_k: int, dtype: torch.dtype) -> dict:
    """The launch plan of a geometry (chunking, shared-memory sizes per kernel,
    workspace bytes), as the library computes it; raises GbtopkError when the
    geometry is refused."""
    out = (ctypes.c_int64 * 13)()
    _check(load_library().gbtopk_plan_query(num_rows, width, top_k, _DTYPES[dtype], out))
    keys = ["chunk", "chunks_per_row", "direct_max", "row_smem", "split", "row_candidates",
            "stream_smem", "final_smem", "workspace_bytes", "ws_row_bytes", "row_smem_sorted",
            "fused", "fused_smem"]
    return dict(zip(keys, list(out)))


def gbtopk_device_status(workspace: torch.Tensor) -> int:
    """Reads and clears the device status word of a workspace (synchronises)."""
    flags = ctypes.c_uint32(0)
    _check(load_library().gbtopk_device_status(_ptr(workspace), ctypes.byref(flags),
                                               _stream_handle(workspace.device)))
    return int(flags.value)


def gbtopk_varlen(logits: torch.Tensor, seq_lens: torch.Tensor, top_k: int,
                  pre_idx: Optional[torch.Tensor], next_n: int, compress_ratio: int,
                  out_indices: torch.Tensor, out_values: Optional[torch.Tensor],
                  deterministic: int, workspace: torch.Tensor, stream=None) -> int:
    """Direct call of the C entry point on tensors (no checks beyond the library's)."""
    R, W = logits.shape
    stride = logits.stride(0) if R > 1 else W
    s = _stream_handle(logits.device) if stream is None else stream
    return _check(load_library().gbtopk_varlen(
        _ptr(logits), _DTYPES[logits.dtype], R, W, stride, _ptr(seq_lens), next_n,
        compress_ratio, top_k, _ptr(pre_idx), _ptr(out_indices), _ptr(out_values),
        int(deterministic), _ptr(workspace), workspace.numel() * workspace.element_size(),
        s))


def gbtopk_varlen_static_ws(logits: torch.Tensor, seq_lens: torch.Tensor, top_k: int,
                            pre_idx: Optional[torch.Tensor], next_n: int, compress_ratio: int,
                            out_indices: torch.Tensor, out_values: Optional[torch.Tensor],
                            deterministic: int, stream=None) -> int:
    """Direct call of the allocation-free variant (library-owned 16 MiB scratch
    per GPU, shared by every call: serialise calls that could overlap)."""
    R, W = logits.shape
    stride = logits.stride(0) if R > 1 else W
    s = _stream_handle(logits.device) if stream is None else stream
    return _check(load_library().gbtopk_varlen_static_ws(
        _ptr(logits), _DTYPES[logits.dtype], R, W, stride, _ptr(seq_lens), next_n,
        compress_ratio, top_k, _ptr(pre_idx), _ptr(out_indices), _ptr(out_values),
        int(deterministic), s))


def gbtopk_page_table_transform(scores: torch.Tensor, lengths: torch.Tensor,
                                row_starts: Optional[torch.Tensor], page_table: torch.Tensor,
                                page_table_row_starts: Optional[torch.Tensor], page_size: int,
                                top_k: int, out: torch.Tensor, out_raw: Optional[torch.Tensor],
                                deterministic: int, workspace: torch.Tensor, stream=None) -> int:
    """Direct call of the C entry point on tensors."""
    R, W = scores.shape
    stride = scores.stride(0) if R > 1 else W
    P = page_table.shape[1]
    pstride = page_table.stride(0) if page_table.shape[0] > 1 else P
    s = _stream_handle(scores.device) if stream is None else stream
    return _check(load_library().gbtopk_page_table_transform(
        _ptr(scores), _DTYPES[scores.dtype], R, W, stride, _ptr(lengths), _ptr(row_starts),
        _ptr(page_table), P, pstride, _ptr(page_table_row_starts), page_size, top_k, _ptr(out),
        _ptr(out_raw), int(deterministic), _ptr(workspace),
        workspace.numel() * workspace.element_size(), s))


def gbtopk_ragged_transform(scores: torch.Tensor, lengths: torch.Tensor,
                            row_starts: Optional[torch.Tensor], topk_indices_offset: torch.Tensor,
                            top_k: int, out: torch.Tensor, deterministic: int,
                            workspace: torch.Tensor, stream=None) -> int:
    """Direct call of the C entry point on tensors."""
    R, W = scores.shape
    stride = scores.stride(0) if R > 1 else W
    s = _stream_handle(scores.device) if stream is None else stream
    return _check(load_library().gbtopk_ragged_transform(
        _ptr(scores), _DTYPES[scores.dtype], R, W, stride, _ptr(lengths), _ptr(row_starts),
        _ptr(topk_indices_offset), top_k, _ptr(out), int(deterministic), _ptr(workspace),
        workspace.numel() * workspace.element_size(), s))


def gbtopk_page_table_transform_cu_seqlens(scores: torch.Tensor, lengths: torch.Tensor,
                                           row_starts: Optional[torch.Tensor],
                                           page_table: torch.Tensor, cu_seqlens_q: torch.Tensor,
                                           top_k: int, out: torch.Tensor, deterministic: int,
                                           workspace: torch.Tensor, stream=None) -> int:
    """Direct call of the C entry point on tensors."""
    R, W = scores.shape
    stride = scores.stride(0) if R > 1 else W
    P = page_table.shape[1]
    pstride = page_table.stride(0) if page_table.shape[0] > 1 else P
    s = _stream_handle(scores.device) if stream is None else stream
    return _check(load_library().gbtopk_page_table_transform_cu_seqlens(
        _ptr(scores), _DTYPES[scores.dtype], R, W, stride, _ptr(lengths), _ptr(row_starts),
        _ptr(page_table), P, pstride, _ptr(cu_seqlens_q), cu_seqlens_q.numel() - 1, top_k,
        _ptr(out), int(deterministic), _ptr(workspace),
        workspace.numel() * workspace.element_size(), s))


# One workspace per (device, stream), grown on demand.  Apart from its
# status word the library writes every workspace byte before reading it, so
# one workspace serves every call on a stream.  Create it (by one eager
# call) before capturing a CUDA graph on that stream.
_WS = {}


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    key = (device.index, _stream_handle(device))
    ws = _WS.get(key)
    if ws is None or ws.numel() < nbytes:
        if torch.cuda.is_current_stream_capturing():
            raise RuntimeError("gbtopk: no workspace for this stream yet; run one eager call "
                               "on the capturing stream before graph capture")
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _WS[key] = ws
    return ws


def _require_cuda(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")


def _out_view(buf: Optional[torch.Tensor], R: int, k: int, dtype, device, name: str):
    if buf is None:
        return torch.empty((R, k), dtype=dtype, device=device)
    if buf.dtype != dtype or buf.device != device or not buf.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor on {device}")
    if tuple(buf.shape) == (R, k):
        return buf
    if buf.dim() == 1 and buf.numel() == R * k:
        return buf.view(R, k)
    raise ValueError(f"{name} must have shape ({R}, {k}) or ({R * k},)")


def top_k_varlen(logits: torch.Tensor, seq_lens: torch.Tensor, top_k: int,
                 pre_idx: Optional[torch.Tensor] = None, compress_ratio: int = 1,
                 next_n: int = 1, return_values: bool = False,
                 out_indices: Optional[torch.Tensor] = None,
                 out_values: Optional[torch.Tensor] = None, deterministic: bool = False,
                 workspace: Optional[torch.Tensor] = None, tie_mode: Optional[str] = None
                 ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Top-k of each row of ``logits`` over its valid columns.

    Row t of request i ranks its first
    ``max(0, (seq_lens[i] - next_n + t + 1) // compress_ratio)`` columns,
    clamped to the width.  Returns ``(indices int32 [R, k], values | None)``;
    unused slots are -1 (values: the dtype's lowest finite value).
    ``deterministic`` orders each row by (value desc, column asc);
    ``tie_mode`` ("small" / "large") fixes which columns equal to the k-th
    value are kept (see ``order_flags``)."""
    flags = order_flags(deterministic, tie_mode)
    _require_cuda(logits, "logits")
    _require_cuda(seq_lens, "seq_lens")
    if logits.dim() != 2 or logits.stride(1) != 1 or logits.dtype not in _DTYPES:
        raise ValueError("logits must be a 2-D fp32/bf16/fp16 tensor with inner stride 1")
    R, W = logits.shape
    if next_n < 1 or R % next_n != 0:
        raise ValueError("num_rows must be a multiple of next_n")
    if seq_lens.dtype != torch.int32 or seq_lens.dim() != 1 or seq_lens.numel() != R // next_n \
            or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 tensor of num_rows // next_n")
    idx = _out_view(out_indices, R, top_k, torch.int32, logits.device, "out_indices")
    val = None
    if return_values:
        val = _out_view(out_values, R, top_k, logits.dtype, logits.device, "out_values")
    hint = None
    if pre_idx is not None:
        ok = (isinstance(pre_idx, torch.Tensor) and pre_idx.device == logits.device
              and pre_idx.dtype == torch.int32 and pre_idx.is_contiguous()
              and tuple(pre_idx.shape) == (R // next_n, top_k))
        if ok:
            hint = pre_idx
        else:
            warnings.warn("pre_idx is malformed and was discarded; running hint-free",
                          RuntimeWarning, stacklevel=2)
    ws = workspace if workspace is not None else _workspace(
        logits.device, gbtopk_workspace_bytes(R, W, top_k, logits.dtype))
    st = gbtopk_varlen(logits, seq_lens, top_k, hint, next_n, compress_ratio, idx, val,
                       flags, ws)
    if st == HINT_DISCARDED:
        warnings.warn("pre_idx is not 16-byte aligned and was discarded; running hint-free",
                      RuntimeWarning, stacklevel=2)
    return idx, val


def top_k_page_table_transform(scores: torch.Tensor, lengths: torch.Tensor,
                               page_table: torch.Tensor, top_k: int, page_size: int = 1,
                               row_starts: Optional[torch.Tensor] = None,
                               page_table_row_starts: Optional[torch.Tensor] = None,
                               out: Optional[torch.Tensor] = None,
                               out_raw_indices: Optional[torch.Tensor] = None,
                               deterministic: bool = False,
                               workspace: Optional[torch.Tensor] = None,
                               tie_mode: Optional[str] = None):
    """Top-k fused with the compact page-table transform.

    Returns ``out`` (physical indices), or ``(out, out_raw_indices)`` when a
    raw-index buffer is given.  ``deterministic`` / ``tie_mode``: as for
    ``top_k_varlen``."""
    flags = order_flags(deterministic, tie_mode)
    for t, name in ((scores, "scores"), (lengths, "lengths"), (page_table, "page_table")):
        _require_cuda(t, name)
    if scores.dim() != 2 or scores.stride(1) != 1 or scores.dtype not in _DTYPES:
        raise ValueError("scores must be a 2-D fp32/bf16/fp16 tensor with inner stride 1")
    R, W = scores.shape
    if page_table.dim() != 2 or page_table.stride(1) != 1 or page_table.dtype != torch.int32 \
            or page_table.shape[0] != R:
        raise ValueError("page_table must be an int32 [num_rows, pt_cols] tensor, inner stride 1")
    for t, name in ((lengths, "lengths"), (row_starts, "row_starts"),
                    (page_table_row_starts, "page_table_row_starts")):
        if t is not None and (t.dtype != torch.int32 or t.numel() != R or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous int32 tensor of num_rows")
    if page_size < 1 or page_size > 2 ** 30:
        raise ValueError("page_size must be in [1, 2**30]")
    if page_size > 1 and row_starts is not None and page_table_row_starts is None:
        raise ValueError("page_table_row_starts is required when page_size > 1 and "
                         "row_starts is given (starts are in different units)")
    o = _out_view(out, R, top_k, torch.int32, scores.device, "out")
    raw = None
    if out_raw_indices is not None:
        raw = _out_view(out_raw_indices, R, top_k, torch.int32, scores.device, "out_raw_indices")
    ws = workspace if workspace is not None else _workspace(
        scores.device, gbtopk_workspace_bytes(R, W, top_k, scores.dtype))
    gbtopk_page_table_transform(scores, lengths, row_starts, page_table, page_table_row_starts,
                                page_size, top_k, o, raw, flags, ws)
    return (o, raw) if raw is not None else o


def _ragged_inputs(scores, lengths, row_starts, name_tensors):
    for t, name in name_tensors:
        _require_cuda(t, name)
    if scores.dim() != 2 or scores.stride(1) != 1 or scores.dtype not in _DTYPES:
        raise ValueError("scores must be a 2-D fp32/bf16/fp16 tensor with inner stride 1")
    R = scores.shape[0]
    for t, name in ((lengths, "lengths"), (row_starts, "row_starts")):
        if t is not None and (t.dtype != torch.int32 or t.numel() != R or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous int32 tensor of num_rows")


def top_k_ragged_transform(scores: torch.Tensor, lengths: torch.Tensor,
                           topk_indices_offset: torch.Tensor, top_k: int,
                           row_starts: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, deterministic: bool = False,
                           workspace: Optional[torch.Tensor] = None,
                           tie_mode: Optional[str] = None) -> torch.Tensor:
    """Top-k fused with the ragged KV index offset (SGLang
    fast_topk_transform_ragged_fused): out = idx + topk_indices_offset[row]."""
    flags = order_flags(deterministic, tie_mode)
    _ragged_inputs(scores, lengths, row_starts,
                   ((scores, "scores"), (lengths, "lengths"),
                    (topk_indices_offset, "topk_indices_offset")))
    R, W = scores.shape
    if (topk_indices_offset.dtype != torch.int32 or topk_indices_offset.numel() != R
            or not topk_indices_offset.is_contiguous()):
        raise ValueError("topk_indices_offset must be a contiguous int32 tensor of num_rows")
    o = _out_view(out, R, top_k, torch.int32, scores.device, "out")
    ws = workspace if workspace is not None else _workspace(
        scores.device, gbtopk_workspace_bytes(R, W, top_k, scores.dtype))
    gbtopk_ragged_transform(scores, lengths, row_starts, topk_indices_offset, top_k, o,
                            flags, ws)
    return o


def top_k_page_table_transform_cu_seqlens(scores: torch.Tensor, lengths: torch.Tensor,
                                          page_table: torch.Tensor, cu_seqlens_q: torch.Tensor,
                                          top_k: int, row_starts: Optional[torch.Tensor] = None,
                                          out: Optional[torch.Tensor] = None,
                                          deterministic: bool = False,
                                          workspace: Optional[torch.Tensor] = None,
                                          tie_mode: Optional[str] = None) -> torch.Tensor:
    """Top-k fused with a page_size-1 page table indexed by request (SGLang
    fast_topk_transform_fused): row r of request b (cu_seqlens_q[b] <= r <
    cu_seqlens_q[b + 1]) gets page_table[b, idx]."""
    flags = order_flags(deterministic, tie_mode)
    _ragged_inputs(scores, lengths, row_starts,
                   ((scores, "scores"), (lengths, "lengths"), (page_table, "page_table"),
                    (cu_seqlens_q, "cu_seqlens_q")))
    R, W = scores.shape
    if page_table.dim() != 2 or page_table.stride(1) != 1 or page_table.dtype != torch.int32:
        raise ValueError("page_table must be an int32 [num_reqs, pt_cols] tensor, inner stride 1")
    if (cu_seqlens_q.dtype != torch.int32 or cu_seqlens_q.dim() != 1
            or cu_seqlens_q.numel() != page_table.shape[0] + 1 or not cu_seqlens_q.is_contiguous()):
        raise ValueError("cu_seqlens_q must be a contiguous int32 tensor of num_reqs + 1")
    o = _out_view(out, R, top_k, torch.int32, scores.device, "out")
    ws = workspace if workspace is not None else _workspace(
        scores.device, gbtopk_workspace_bytes(R, W, top_k, scores.dtype))
    gbtopk_page_table_transform_cu_seqlens(scores, lengths, row_starts, page_table, cu_seqlens_q,
                                           top_k, o, flags, ws)
    return o
