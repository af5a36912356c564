"""Host-side tests of the C ABI: no GPU needed, nothing is enqueued.

* the library loads and exports every function declared in include/gbtopk.h;
* argument checks return the documented negative status before any CUDA call
  (pointers here are never dereferenced: every call fails validation);
* the launch plan is total over the supported envelope and consistent
  (a fuzz in the spirit of the route-totality sweeps of TensorRT-LLM PR #17821).
"""
import ctypes
import os
import random
import re

import pytest
import torch

import sparse_attention_top_gb300 as gb

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gbtopk.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gbtopk_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol():
    names = _declared()
    assert {"gbtopk_varlen", "gbtopk_page_table_transform", "gbtopk_workspace_bytes",
            "gbtopk_status_str"} <= set(names)
    lib = ctypes.CDLL(gb.library_path())
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gbtopk.h but not exported"


def test_status_strings():
    for code in (0, 1, -1, -2, -3, -4, -5, -6, -7):
        s = gb.gbtopk_status_str(code)
        assert s.startswith("GBTOPK_")
    assert "unknown" in gb.gbtopk_status_str(42)


# fake, never-dereferenced device addresses (every call below fails first)
A = 0x10000000
WS = 0x20000000


def _varlen(**kw):
    lib = gb.load_library()
    a = dict(logits=A, dtype=0, num_rows=4, width=100, row_stride=100, seq_lens=A + 4096,
             next_n=1, cr=1, top_k=8, pre_idx=None, out=A + 8192, out_values=None, det=0,
             ws=WS, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return lib.gbtopk_varlen(a["logits"], a["dtype"], a["num_rows"], a["width"], a["row_stride"],
                             a["seq_lens"], a["next_n"], a["cr"], a["top_k"], a["pre_idx"],
                             a["out"], a["out_values"], a["det"], a["ws"], a["ws_bytes"],
                             a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(next_n=0), gb.EINVAL),
    (dict(next_n=3), gb.EINVAL),            # 4 rows not a multiple of 3
    (dict(cr=0), gb.EINVAL),
    (dict(top_k=0), gb.EINVAL),
    (dict(top_k=gb.MAX_TOP_K + 1), gb.EUNSUPPORTED),
    (dict(dtype=7), gb.EINVAL),
    (dict(num_rows=-1), gb.EINVAL),
    (dict(row_stride=50), gb.EINVAL),       # stride below the width
    (dict(out=None), gb.EINVAL),
    (dict(logits=None), gb.EINVAL),
    (dict(seq_lens=None), gb.EINVAL),
    (dict(logits=A + 2), gb.EALIGN),        # fp32 scores must be 4-byte aligned
    (dict(out=A + 8196), gb.EALIGN),        # outputs 16-byte aligned
    (dict(out_values=A + 65540), gb.EALIGN),
    (dict(out_values=A + 8192 + 64), gb.EOVERLAP),
    (dict(ws=None), gb.EWORKSPACE),
    (dict(ws=WS + 16), gb.EWORKSPACE),      # workspace 256-byte aligned
    (dict(ws_bytes=16), gb.EWORKSPACE),
    (dict(det=gb.TIE_SMALL | gb.TIE_LARGE), gb.EINVAL),   # the tie modes exclude each other
    (dict(det=gb.SORTED | gb.TIE_SMALL | gb.TIE_LARGE), gb.EINVAL),
    (dict(det=8), gb.EINVAL),                          # unknown flag
    (dict(det=-1), gb.EINVAL),
])
def test_varlen_argument_checks(kw, status):
    assert _varlen(**kw) == status


@pytest.mark.parametrize("det", [gb.SORTED | gb.TIE_SMALL | gb.TIE_LARGE, 16])
def test_order_flags_checked_by_every_entry(det):
    assert _pt(det=det) == gb.EINVAL
    assert _ragged(det=det) == gb.EINVAL
    assert _cu(det=det) == gb.EINVAL


def test_order_flags_mapping():
    assert gb.order_flags() == 0
    assert gb.order_flags(True) == gb.SORTED == 1   # the sorted order alone keeps its meaning
    assert gb.order_flags(False, "small") == gb.TIE_SMALL
    assert gb.order_flags(False, "large") == gb.TIE_LARGE
    assert gb.order_flags(True, "large") == gb.SORTED | gb.TIE_LARGE
    with pytest.raises(ValueError):
        gb.order_flags(False, "middle")


def test_zero_rows_is_a_noop():
    assert _varlen(num_rows=0, logits=None, out=None, seq_lens=None, ws=None) == gb.OK


def _pt(**kw):
    lib = gb.load_library()
    a = dict(scores=A, dtype=0, num_rows=2, width=64, row_stride=64, lengths=A + 4096,
             row_starts=None, page_table=A + 8192, pt_cols=16, pt_row_stride=16,
             pt_row_starts=None, page_size=4, top_k=8, out=A + 16384, out_raw=A + 32768, det=1,
             ws=WS, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return lib.gbtopk_page_table_transform(
        a["scores"], a["dtype"], a["num_rows"], a["width"], a["row_stride"], a["lengths"],
        a["row_starts"], a["page_table"], a["pt_cols"], a["pt_row_stride"], a["pt_row_starts"],
        a["page_size"], a["top_k"], a["out"], a["out_raw"], a["det"], a["ws"], a["ws_bytes"],
        a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(page_size=0), gb.EINVAL),
    (dict(page_size=(1 << 30) + 1), gb.EINVAL),
    (dict(row_starts=A + 4160), gb.EINVAL),   # page_size > 1, row_starts, no pt starts
    (dict(page_table=None), gb.EINVAL),
    (dict(lengths=None), gb.EINVAL),
    (dict(pt_row_stride=8), gb.EINVAL),
    (dict(out_raw=A + 16384 + 32), gb.EOVERLAP),
    (dict(out_raw=A + 32772), gb.EALIGN),
    (dict(top_k=gb.MAX_TOP_K + 1), gb.EUNSUPPORTED),
    (dict(ws_bytes=0), gb.EWORKSPACE),
])
def test_page_table_argument_checks(kw, status):
    assert _pt(**kw) == status


def test_plan_totality_and_consistency():
    rnd = random.Random(3)
    dts = [torch.float32, torch.bfloat16, torch.float16]
    widths = [1, 7, 32, 2047, 2048, 4096, 8191, 8192, 8193, 16384, 16385, 65536, 131075,
              131076, 163840, 262144, 1 << 20]
    for trial in range(3000):
        R = rnd.choice([1, 2, 4, 16, 64, 256, 1024, 4096, rnd.randint(1, 5000)])
        W = rnd.choice(widths + [rnd.randint(1, 1 << 19)])
        k = rnd.choice([1, 2, 64, 512, 1024, 2048, rnd.randint(1, 2048), 2049, 4096, 16384,
                        rnd.randint(1, gb.MAX_TOP_K)])
        dt = rnd.choice(dts)
        p = gb.gbtopk_plan_query(R, W, k, dt)
        es = 4 if dt == torch.float32 else 2
        # two-kernel (fused) split path up to top_k 2048 and the three-kernel
        # path above it, both with 64 KB chunks
        fused_slots = R * -(-W * es // 65536)
        assert p["fused"] == int(bool(p["split"]) and k <= 2048 and fused_slots <= 2048)
        assert p["chunk"] * es == 65536
        for key in ("row_smem", "row_smem_sorted", "stream_smem", "final_smem", "fused_smem"):
            assert p[key] <= 227 * 1024
        assert p["row_smem_sorted"] >= p["row_smem"]
        if p["fused"]:      # three chunk blocks per SM
            assert 3 * (p["fused_smem"] + 1024) <= 228 * 1024
            assert p["stream_smem"] == 0 and p["final_smem"] == 0
        # on small batches a stream block and a row block fit on one SM together
        elif p["split"] and R <= 128:
            assert p["row_smem"] + p["stream_smem"] + 2048 <= 228 * 1024
        if p["split"]:
            assert W > 65536 // es and p["direct_max"] == k
            assert p["chunk"] * p["chunks_per_row"] >= W and p["chunks_per_row"] <= 256
            assert p["row_candidates"] >= k and p["ws_row_bytes"] >= 8 * p["row_candidates"]
        else:
            assert p["direct_max"] == W and p["chunks_per_row"] == 1 and p["ws_row_bytes"] == 0
        assert p["workspace_bytes"] == gb.gbtopk_workspace_bytes(R, W, k, dt) == \
            256 + R * p["ws_row_bytes"]
    with pytest.raises(gb.GbtopkError):
        gb.gbtopk_plan_query(4, 100, 0, torch.float32)
    assert gb.gbtopk_workspace_bytes(4, 100, 0, torch.float32) == 0


def test_no_cpu_path():
    x = torch.randn(2, 64)
    with pytest.raises(ValueError):
        gb.top_k_varlen(x, torch.tensor([64, 64], dtype=torch.int32), 8)


def _ragged(**kw):
    lib = gb.load_library()
    a = dict(scores=A, dtype=0, num_rows=2, width=64, row_stride=64, lengths=A + 4096,
             row_starts=None, offsets=A + 8192, top_k=8, out=A + 16384, det=0, ws=WS,
             ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return lib.gbtopk_ragged_transform(
        a["scores"], a["dtype"], a["num_rows"], a["width"], a["row_stride"], a["lengths"],
        a["row_starts"], a["offsets"], a["top_k"], a["out"], a["det"], a["ws"], a["ws_bytes"],
        a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(offsets=None), gb.EINVAL),
    (dict(lengths=None), gb.EINVAL),
    (dict(out=A + 16388), gb.EALIGN),
    (dict(top_k=gb.MAX_TOP_K + 1), gb.EUNSUPPORTED),
    (dict(ws_bytes=0), gb.EWORKSPACE),
])
def test_ragged_argument_checks(kw, status):
    assert _ragged(**kw) == status


def _cu(**kw):
    lib = gb.load_library()
    a = dict(scores=A, dtype=0, num_rows=3, width=64, row_stride=64, lengths=A + 4096,
             row_starts=None, page_table=A + 8192, pt_cols=16, pt_row_stride=16,
             cu=A + 12288, num_reqs=2, top_k=8, out=A + 16384, det=0, ws=WS, ws_bytes=1 << 20,
             stream=None)
    a.update(kw)
    return lib.gbtopk_page_table_transform_cu_seqlens(
        a["scores"], a["dtype"], a["num_rows"], a["width"], a["row_stride"], a["lengths"],
        a["row_starts"], a["page_table"], a["pt_cols"], a["pt_row_stride"], a["cu"],
        a["num_reqs"], a["top_k"], a["out"], a["det"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(cu=None), gb.EINVAL),
    (dict(page_table=None), gb.EINVAL),
    (dict(num_reqs=-1), gb.EINVAL),
    (dict(pt_row_stride=8), gb.EINVAL),
    (dict(out=A + 16388), gb.EALIGN),
    (dict(ws=None), gb.EWORKSPACE),
])
def test_cu_seqlens_argument_checks(kw, status):
    assert _cu(**kw) == status


@pytest.mark.parametrize("num_rows,width,top_k,dtype,status", [
    (4, 1 << 31, 8, 0, gb.EUNSUPPORTED),          # width beyond the plan (int32 columns)
    (4, 100, 0, 0, gb.EINVAL),
    (4, 100, gb.MAX_TOP_K + 1, 0, gb.EUNSUPPORTED),
    (4, 100, 8, 7, gb.EINVAL),                    # unknown dtype
    (4, 4 * 16384 * 256 + 1, 8, 0, gb.EUNSUPPORTED),  # wider than the split plan allows
    (1024, 262144, 2048, 0, gb.EWORKSPACE),       # more scratch than the built-in buffer
])
def test_static_scratch_refusals_match_the_plan(num_rows, width, top_k, dtype, status):
    """The allocation-free entry point refuses a geometry before touching the
    device, with the status gbtopk_varlen's plan gives (or EWORKSPACE when
    the built-in scratch is too small)."""
    lib = gb.load_library()
    st = lib.gbtopk_varlen_static_ws(A, dtype, num_rows, width, width, A + 4096, 1, 1, top_k, None,
                                     A + 8192, None, 0, None)
    assert st == status
    if status != gb.EWORKSPACE:
        assert _varlen(num_rows=num_rows, width=width, row_stride=width, top_k=top_k,
                       dtype=dtype) == status
