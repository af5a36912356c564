"""Comparison of the CUDA path with the oracle (tie-aware; bit-exact when
deterministic).  Acceptance per row, following the exactness definition of
TensorRT-LLM PR #17821 ("tie-aware exactness using signed-zero-normalized
value-multiset comparison"):

* the -1 pattern is identical (min(k, n) live slots, then -1);
* live indices are unique and inside [0, n);
* the multiset of selected values equals the oracle's at tolerance 0, with
  -0.0 and +0.0 identified;
* returned values are bit copies of logits[idx]; padding holds the lowest
  finite value of the dtype;
* deterministic mode: the index list is bit-identical to the oracle's;
* a tie mode without the sorted order: the selected index set is the
  oracle's (the set is unique once the tie mode fixes which of the values
  equal to the k-th are kept; the order is not).
"""
from __future__ import annotations

import torch

LOWEST_BITS = {torch.float32: -8388609,  # 0xFF7FFFFF as int32
               torch.bfloat16: -129,     # 0xFF7F as int16
               torch.float16: -1025}     # 0xFBFF as int16
INT_VIEW = {torch.float32: torch.int32, torch.bfloat16: torch.int16, torch.float16: torch.int16}


def _norm(v: torch.Tensor) -> torch.Tensor:
    v = v.double()
    return torch.where(v == 0, torch.zeros_like(v), v)


def check_rows(logits_cpu: torch.Tensor, n_rows, top_k: int, gpu_idx: torch.Tensor,
               ref_idx: torch.Tensor, gpu_val=None, deterministic: bool = False,
               rows=None, col0=None, same_set: bool = False) -> None:
    """Asserts parity for the given rows (all by default).

    ``logits_cpu`` is the [R, W] score matrix, ``n_rows[r]`` the valid count
    and ``col0[r]`` the column of local index 0 (page-table row starts)."""
    gi = gpu_idx.cpu()
    ri = ref_idx.cpu()
    gv = gpu_val.cpu() if gpu_val is not None else None
    R = gi.shape[0]
    rows = range(R) if rows is None else rows
    for r in rows:
        n = int(n_rows[r])
        c0 = 0 if col0 is None else int(col0[r])
        m = min(n, top_k)
        g = gi[r]
        assert bool((g[m:] == -1).all()), f"row {r}: -1 padding pattern differs"
        live = g[:m].long()
        assert bool((live >= 0).all()) and bool((live < n).all()), f"row {r}: index out of range"
        assert torch.unique(live).numel() == m, f"row {r}: duplicate indices"
        if deterministic:
            assert torch.equal(g, ri[r]), f"row {r}: deterministic index list differs"
        if same_set:
            assert torch.equal(torch.sort(live).values, torch.sort(ri[r][:m].long()).values), \
                f"row {r}: selected index set differs"
        row = logits_cpu[r, c0:c0 + n]
        got = torch.sort(_norm(row[live]), descending=True).values
        ref = torch.sort(_norm(row[ri[r][:m].long()]), descending=True).values
        assert torch.equal(got, ref), f"row {r}: selected value multiset differs"
        if gv is not None:
            iv = INT_VIEW[logits_cpu.dtype]
            assert torch.equal(gv[r][:m].view(iv), row[live].contiguous().view(iv)), \
                f"row {r}: values are not bit copies of logits[idx]"
            assert bool((gv[r][m:].view(iv) == LOWEST_BITS[logits_cpu.dtype]).all()), \
                f"row {r}: value padding is not the lowest finite value"
