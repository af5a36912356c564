"""Seeded synthetic inputs for the DSA indexer top-K workloads.

Shared by the tests, the benchmark and the smoke check.  This module holds
none of the selection method's arithmetic: it only draws random tensors with
the shapes, value distributions and length mixes of the workloads described
on the pages (FlashInfer `top_k_varlen` docs; TensorRT-LLM PR #17821
benchmark and test sections; SGLang PR #33237 for the compact page table).
The pages measure on real decode captures that are not available here; these
seeded tensors stand in for them.

Every tensor is created on the CPU with its own ``torch.Generator`` seeded
as ``config_id * 1000 + variant`` so a case is reproducible byte for byte.

The previous-step hint ``pre_idx`` is synthesised the way the workloads
describe it (the top-k columns of a "previous" row, strongest first): it is
input data, and the selection never depends on it.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class VarlenCase:
    """Inputs of one `top_k_varlen` call (all CPU tensors)."""
    name: str
    logits: torch.Tensor            # [num_rows, width] (inner stride 1)
    seq_lens: torch.Tensor          # int32 [num_rows // next_n], KV-token units
    top_k: int
    next_n: int = 1
    compress_ratio: int = 1
    pre_idx: Optional[torch.Tensor] = None   # int32 [num_rows // next_n, top_k]
    return_values: bool = False
    deterministic: bool = False
    info: dict = field(default_factory=dict)


@dataclass
class PageTableCase:
    """Inputs of one fused top-k + compact page-table transform call."""
    name: str
    scores: torch.Tensor            # [num_rows, width] view with a row stride
    lengths: torch.Tensor           # int32 [num_rows]
    row_starts: Optional[torch.Tensor]
    page_table: torch.Tensor        # int32 [num_rows, pt_cols] (inner stride 1)
    page_table_row_starts: Optional[torch.Tensor]
    page_size: int
    top_k: int
    deterministic: bool = True
    info: dict = field(default_factory=dict)


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _hint_from(prev: torch.Tensor, cols: torch.Tensor, top_k: int) -> torch.Tensor:
    """Top-k columns of each row of ``prev`` among its first ``cols[i]``
    columns, strongest first (argmax in slot 0); short rows pad with -1."""
    n_req = prev.shape[0]
    hint = torch.full((n_req, top_k), -1, dtype=torch.int32)
    for i in range(n_req):
        c = int(cols[i])
        if c <= 0:
            continue
        m = min(top_k, c)
        hint[i, :m] = torch.topk(prev[i, :c].float(), m, sorted=True).indices.to(torch.int32)
    return hint


def tiny(seed: int = 1000) -> VarlenCase:
    """4 rows x 4096 fp32 ~N(0,1); seq_lens ~U[1,6000] with one row forced to
    0 and one forced above the width; top_k=512; values returned."""
    g = _gen(seed)
    R, W = 4, 4096
    logits = torch.randn(R, W, generator=g)
    seq = torch.randint(1, 6001, (R,), generator=g, dtype=torch.int64)
    seq[3] = 0
    if not bool((seq > W).any()):
        seq[0] = int(torch.randint(W + 1, 6001, (1,), generator=g))
    return VarlenCase("tiny", logits, seq.to(torch.int32), 512, return_values=True,
                      info={"config": 0})


def dsv32_decode(rows: int = 64, width: int = 163840, top_k: int = 2048,
                 hinted: bool = True, seed: int = 2000,
                 min_len: Optional[int] = None) -> VarlenCase:
    """DSv3.2-like decode: N(0,1) with +4 on 1% of the columns of each row,
    quantised to 1/64 (ties); the hint is the top-k of the row before a
    N(0,0.3) perturbation; seq_lens ~U[2048, width]."""
    g = _gen(seed)
    base = torch.randn(rows, width, generator=g)
    n_boost = max(1, width // 100)
    for r in range(rows):
        cols = torch.randperm(width, generator=g)[:n_boost]
        base[r, cols] += 4.0
    prev = torch.round(base * 64.0) / 64.0
    lo = 2048 if min_len is None else min_len
    seq = torch.randint(lo, width + 1, (rows,), generator=g, dtype=torch.int64)
    noise = torch.randn(rows, width, generator=g) * 0.3
    logits = torch.round((prev + noise) * 64.0) / 64.0
    hint = _hint_from(prev, torch.clamp(seq, max=width), top_k) if hinted else None
    return VarlenCase("dsv32_decode", logits, seq.to(torch.int32), top_k, pre_idx=hint,
                      info={"config": 1, "hinted": hinted})


def long_row_sweep(rows: int, top_k: int, hinted: bool, width: int = 262144,
                   seed: Optional[int] = None) -> VarlenCase:
    """Long-row batch: N(0,1) plus a per-row offset ~N(0,2);
    seq_lens ~U[width/2, width]; hint from the row before a N(0,0.3) noise."""
    if seed is None:
        seed = 3000 + rows % 997 + {512: 0, 1024: 1, 2048: 2}.get(top_k, 3) * 100
    g = _gen(seed)
    base = torch.randn(rows, width, generator=g)
    base += torch.randn(rows, 1, generator=g) * 2.0
    seq = torch.randint(width // 2, width + 1, (rows,), generator=g, dtype=torch.int64)
    logits = base + torch.randn(rows, width, generator=g) * 0.3
    hint = _hint_from(base, torch.clamp(seq, max=width), top_k) if hinted else None
    return VarlenCase(f"long_row_sweep_r{rows}_k{top_k}", logits, seq.to(torch.int32), top_k,
                      pre_idx=hint, info={"config": 2, "hinted": hinted})


def dsv4_mtp(hinted: bool = False, requests: int = 128, width: int = 65536,
             top_k: int = 1024, seed: int = 4000) -> VarlenCase:
    """DSv4-like MTP: next_n=4, compress_ratio=4, bf16 N(0,1) logits;
    seq_lens ~U[0, 4*width] in KV tokens with four requests forced to 0..3."""
    g = _gen(seed)
    next_n, cr = 4, 4
    R = requests * next_n
    base = torch.randn(R, width, generator=g)
    logits = (base + torch.randn(R, width, generator=g) * 0.3).to(torch.bfloat16)
    seq = torch.randint(0, cr * width + 1, (requests,), generator=g, dtype=torch.int64)
    forced = torch.randperm(requests, generator=g)[:4]
    for v, i in enumerate(forced.tolist()):
        seq[i] = v
    hint = None
    if hinted:
        last_rows = base.view(requests, next_n, width)[:, next_n - 1, :]
        hint = _hint_from(last_rows, torch.clamp(seq // cr, max=width), top_k)
    return VarlenCase("dsv4_mtp", logits, seq.to(torch.int32), top_k, next_n=next_n,
                      compress_ratio=cr, pre_idx=hint, info={"config": 3, "hinted": hinted})


def short_rows(rows: int = 4096, width: int = 2048, top_k: int = 512,
               seed: int = 4100) -> VarlenCase:
    """Short rows: fp16 N(0,1), seq_lens ~U[1, width], top_k=512."""
    g = _gen(seed)
    logits = torch.randn(rows, width, generator=g).to(torch.float16)
    seq = torch.randint(1, width + 1, (rows,), generator=g, dtype=torch.int32)
    return VarlenCase("short_rows", logits, seq, top_k, info={"config": 3})


def page_table_case(rows: int = 256, width: int = 32768, row_stride: int = 33024,
                    page_size: int = 64, pt_cols: int = 1024, top_k: int = 2048,
                    deterministic: bool = True, seed: int = 5000) -> PageTableCase:
    """Compact page table: fp32 scores with padding between rows (the gap
    holds 3e38), ragged lengths ~U[1,width] and row starts, page_table int32
    ~U[0,1e6), page_table_row_starts in entries."""
    g = _gen(seed)
    storage = torch.full((rows, row_stride), 3.0e38)
    storage[:, :width] = torch.randn(rows, width, generator=g)
    scores = storage[:, :width]
    lengths = torch.randint(1, width + 1, (rows,), generator=g, dtype=torch.int64)
    row_starts = torch.stack([torch.randint(0, width - int(L) + 1, (1,), generator=g)[0]
                              for L in lengths])
    page_table = torch.randint(0, 1_000_000, (rows, pt_cols), generator=g, dtype=torch.int32)
    pages_used = (lengths - 1) // page_size + 1
    pt_starts = torch.stack([torch.randint(0, pt_cols - int(p) + 1, (1,), generator=g)[0]
                             for p in pages_used])
    return PageTableCase("page_table", scores, lengths.to(torch.int32),
                         row_starts.to(torch.int32), page_table, pt_starts.to(torch.int32),
                         page_size, top_k, deterministic=deterministic,
                         info={"config": 4})
