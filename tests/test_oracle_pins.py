"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

The oracle must not be trusted on its own word, so it is checked here
against (1) hand-worked golden cases under ``tests/golden/`` (row-length
formula, selection order with signed zeros / infinities / denormals, short
row padding, the compact page-table formula), (2) brute force on tiny rows
in pure Python, (3) a library routine (``torch.topk`` value multiset),
(4) invariants on the workload generators, and (5) mutation tests: textual
mutants of the oracle source (a dropped term, a flipped sign, a transposed
operand) are compiled and must each fail at least one pin.
"""
import ctypes
import json
import os
import random
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "topk_oracle.c")
DT = {"float32": (torch.float32, 0), "bfloat16": (torch.bfloat16, 1), "float16": (torch.float16, 2)}


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bind(lib):
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.oracle_row_length.restype = i64
    lib.oracle_row_length.argtypes = [i64, i64, i64, i64, i64]
    lib.oracle_select_row.restype = ctypes.c_int
    lib.oracle_select_row.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp]
    lib.oracle_page_table_transform.restype = ctypes.c_int
    lib.oracle_page_table_transform.argtypes = [
        vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, i64, i64, vp, i32, i32, vp, vp]
    lib.oracle_ragged_offset_transform.restype = ctypes.c_int
    lib.oracle_ragged_offset_transform.argtypes = [
        vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, i32, vp]
    lib.oracle_select_row_large_ties.restype = ctypes.c_int
    lib.oracle_select_row_large_ties.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp]
    lib.oracle_seqs_page_table_transform.restype = ctypes.c_int
    lib.oracle_seqs_page_table_transform.argtypes = [
        vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, i64, i64, vp, i64, i32, vp]
    return lib


def _row_tensor(case):
    if case["dtype"] == "float32":
        u = [int(h, 16) for h in case["row_f32_hex"]]
        return torch.tensor(np.array(u, dtype=np.uint32).view(np.float32))
    u = [int(h, 16) for h in case["row_u16_hex"]]
    t = torch.tensor(np.array(u, dtype=np.uint16).view(np.int16))
    return t.view(DT[case["dtype"]][0])


def _bits(t):
    if t.dtype == torch.float32:
        return [format(int(x), "08x") for x in t.view(torch.int32).numpy().view(np.uint32)]
    return [format(int(x), "04x") for x in t.view(torch.int16).numpy().view(np.uint16)]


def golden_failures(lib):
    """Run every golden pin through ``lib``; return a list of failure strings."""
    fails = []
    g = _golden("row_lengths.json")
    for seq, nn, cr, w, expect in g["cases"]:
        got = [lib.oracle_row_length(seq, nn, t, cr, w) for t in range(nn)]
        if got != expect:
            fails.append(f"row_length{(seq, nn, cr, w)}: {got} != {expect}")
    for case in _golden("selection.json")["cases"]:
        row = _row_tensor(case)
        k = case["k"]
        idx = torch.empty(k, dtype=torch.int32)
        val = torch.empty(k, dtype=row.dtype)
        rc = lib.oracle_select_row(row.data_ptr(), DT[case["dtype"]][1], case["n"], k,
                                   idx.data_ptr(), val.data_ptr())
        if rc != 0 or idx.tolist() != case["indices"] or _bits(val) != case["values_hex"]:
            fails.append(f"select {case['name']}: rc={rc} {idx.tolist()} {_bits(val)}")
    for case in _golden("page_table.json")["cases"]:
        W = case["width"]
        if "scores" in case:
            scores = torch.tensor(case["scores"], dtype=torch.float32)
        else:
            scores = torch.zeros(W)
            for c, v in case["nonzero_scores"].items():
                scores[int(c)] = v
        scores = scores.view(1, W)
        pt = torch.tensor([case["page_table_row"]], dtype=torch.int32)
        lengths = torch.tensor([case["length"]], dtype=torch.int32)
        rs = None if case["row_start"] is None else torch.tensor([case["row_start"]], dtype=torch.int32)
        prs = (None if case["page_table_row_start"] is None
               else torch.tensor([case["page_table_row_start"]], dtype=torch.int32))
        k = case["k"]
        out = torch.empty(k, dtype=torch.int32)
        raw = torch.empty(k, dtype=torch.int32)
        rc = lib.oracle_page_table_transform(
            scores.data_ptr(), 0, 1, W, W, lengths.data_ptr(),
            rs.data_ptr() if rs is not None else None, pt.data_ptr(), pt.shape[1], pt.shape[1],
            prs.data_ptr() if prs is not None else None, case["page_size"], k,
            out.data_ptr(), raw.data_ptr())
        if rc != 0 or out.tolist() != case["out"] or raw.tolist() != case["out_raw"]:
            fails.append(f"page_table {case['name']}: rc={rc} {out.tolist()} {raw.tolist()}")
    for case in _golden("ties.json")["cases"]:
        row = torch.tensor(case["row"], dtype=torch.float32)
        k = case["k"]
        for mode, fn in (("small", lib.oracle_select_row), ("large", lib.oracle_select_row_large_ties)):
            idx = torch.empty(k, dtype=torch.int32)
            rc = fn(row.data_ptr(), 0, row.numel(), k, idx.data_ptr(), None)
            if rc != 0 or idx.tolist() != case[mode]:
                fails.append(f"ties {case['name']} {mode}: rc={rc} {idx.tolist()}")
    ep = _golden("epilogues.json")
    for case in ep["ragged"]:
        scores = torch.tensor([case["scores"]], dtype=torch.float32)
        W = scores.shape[1]
        lengths = torch.tensor([case["length"]], dtype=torch.int32)
        rs = None if case["row_start"] is None else torch.tensor([case["row_start"]], dtype=torch.int32)
        off = torch.tensor([case["offset"]], dtype=torch.int32)
        k = case["k"]
        out = torch.empty(k, dtype=torch.int32)
        rc = lib.oracle_ragged_offset_transform(
            scores.data_ptr(), 0, 1, W, W, lengths.data_ptr(),
            rs.data_ptr() if rs is not None else None, off.data_ptr(), k, out.data_ptr())
        if rc != 0 or out.tolist() != case["out"]:
            fails.append(f"ragged {case['name']}: rc={rc} {out.tolist()}")
    for case in ep["requests"]:
        scores = torch.tensor(case["scores"], dtype=torch.float32)
        R, W = scores.shape
        lengths = torch.tensor(case["lengths"], dtype=torch.int32)
        cu = torch.tensor(case["cu_seqlens_q"], dtype=torch.int32)
        pt = torch.tensor(case["page_table"], dtype=torch.int32)
        rs = (torch.tensor(case["row_starts"], dtype=torch.int32) if case.get("row_starts") is not None
              else None)
        k = case["k"]
        out = torch.empty(R, k, dtype=torch.int32)
        rc = lib.oracle_seqs_page_table_transform(
            scores.data_ptr(), 0, R, W, W, lengths.data_ptr(),
            rs.data_ptr() if rs is not None else None, pt.data_ptr(), pt.shape[1],
            pt.shape[1], cu.data_ptr(), cu.numel() - 1, k, out.data_ptr())
        if rc != 0 or out.tolist() != case["out"]:
            fails.append(f"requests {case['name']}: rc={rc} {out.tolist()}")
    return fails


def test_golden_pins(oracle_mod):
    lib = _bind(oracle_mod._load())
    assert golden_failures(lib) == []


def test_page_table_requires_explicit_pt_starts(oracle_mod):
    # page_size > 1 with row_starts but no page_table_row_starts is refused
    # (starts are in different units: score elements vs page-table entries).
    scores = torch.zeros(1, 8)
    with pytest.raises(ValueError):
        oracle_mod.page_table_transform(scores, torch.tensor([4], dtype=torch.int32),
                                        torch.zeros(1, 4, dtype=torch.int32), 2, page_size=4,
                                        row_starts=torch.tensor([1], dtype=torch.int32))


def _brute(values, n, k):
    order = sorted(range(n), key=lambda j: (-values[j], j))
    return order[:k] + [-1] * (k - min(k, n))


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "float16"])
def test_brute_force_tiny_rows(oracle_mod, dtype):
    rnd = random.Random(7)
    specials = [float("-inf"), -1.0, -0.0, 0.0, 1e-45, 2.0 ** -24, 1.0, 3.0, float("inf")]
    tdt = DT[dtype][0]
    for trial in range(300):
        n_alloc = rnd.randint(1, 24)
        vals = [rnd.choice(specials) if rnd.random() < 0.7 else rnd.uniform(-4, 4)
                for _ in range(n_alloc)]
        row = torch.tensor(vals, dtype=torch.float64).to(tdt)
        exact = [float(x) for x in row.double().tolist()]
        n = rnd.randint(0, n_alloc)
        for k in range(1, n_alloc + 3):
            idx, val = oracle_mod.select_row(row, n, k)
            assert idx.tolist() == _brute(exact, n, k), (dtype, exact, n, k)


def test_torch_topk_value_multiset(oracle_mod):
    g = torch.Generator().manual_seed(11)
    for trial in range(20):
        n = int(torch.randint(1, 6000, (1,), generator=g))
        row = torch.randn(n, generator=g)
        if trial % 2:
            row = torch.round(row * 8) / 8   # force ties
        for k in (1, 7, 512, 2048):
            idx, val = oracle_mod.select_row(row, n, k)
            m = min(n, k)
            ref = torch.topk(row.double(), m).values
            assert torch.equal(val[:m].double(), ref)
            assert torch.equal(row[idx[:m].long()], val[:m])


def check_invariants(logits, n_rows, top_k, idx, val=None):
    """Selection invariants that hold for any exact top-k, any size."""
    for r in range(logits.shape[0]):
        n = int(n_rows[r])
        row = logits[r, :n].double()
        sel = idx[r]
        m = min(n, top_k)
        assert int((sel >= 0).sum()) == m
        assert bool((sel[m:] == -1).all()) and bool((sel[:m] >= 0).all())
        s = sel[:m].long()
        assert bool((s < n).all())
        assert len(set(s.tolist())) == m
        if m < n:
            mask = torch.ones(n, dtype=torch.bool)
            mask[s] = False
            assert float(row[s].min()) >= float(row[mask].max())
        else:
            assert sorted(s.tolist()) == list(range(n))
        if val is not None:
            assert torch.equal(val[r, :m], logits[r, s])


def test_invariants_on_workloads(oracle_mod):
    cases = [workloads.tiny(),
             workloads.short_rows(rows=64),
             workloads.dsv4_mtp(requests=8, width=4096, top_k=256),
             workloads.dsv32_decode(rows=4, width=16384, top_k=512)]
    for c in cases:
        R = c.logits.shape[0]
        idx, val = oracle_mod.topk_varlen(c.logits, c.seq_lens, c.top_k, c.next_n,
                                          c.compress_ratio, return_values=True)
        n_rows = oracle_mod.row_lengths(c.seq_lens.tolist(), R, c.next_n, c.compress_ratio,
                                        c.logits.shape[1])
        check_invariants(c.logits, n_rows, c.top_k, idx, val)
        # the batch entry agrees with the single-row entry
        for r in range(R):
            i1, v1 = oracle_mod.select_row(c.logits[r], int(n_rows[r]), c.top_k)
            assert torch.equal(i1, idx[r]) and torch.equal(v1.view(-1), val[r])


def test_tiny_case_shape(oracle_mod):
    c = workloads.tiny()
    n = oracle_mod.row_lengths(c.seq_lens.tolist(), 4, 1, 1, 4096)
    assert 0 in n.tolist() and 4096 in n.tolist()   # an empty row and a clamped row
    idx, _ = oracle_mod.topk_varlen(c.logits, c.seq_lens, 512)
    assert bool((idx[3] == -1).all())


def test_strided_view_matches_compact(oracle_mod):
    c = workloads.page_table_case(rows=6, width=2048, row_stride=2100, pt_cols=64,
                                  top_k=300, page_size=64)
    out1, raw1 = oracle_mod.page_table_transform(c.scores, c.lengths, c.page_table, c.top_k,
                                                 c.page_size, c.row_starts,
                                                 c.page_table_row_starts)
    out2, raw2 = oracle_mod.page_table_transform(c.scores.contiguous(), c.lengths,
                                                 c.page_table, c.top_k, c.page_size,
                                                 c.row_starts, c.page_table_row_starts)
    assert torch.equal(out1, out2) and torch.equal(raw1, raw2)


MUTANTS = [
    ("control: unmodified source", "", ""),
    ("dropped +1 in numerator", "int64_t num = seq_len - next_n + t + 1;",
     "int64_t num = seq_len - next_n + t;"),
    ("missing width clamp", "return n < width ? n : width;", "return n;"),
    ("ascending order", "if (x->v > y->v)\n        return -1;\n    if (x->v < y->v)\n        return 1;\n"
                        "    return (x->j < y->j)",
     "if (x->v > y->v)\n        return 1;\n    if (x->v < y->v)\n        return -1;\n"
     "    return (x->j < y->j)"),
    ("tie order reversed", "return (x->j < y->j) ? -1 : (x->j > y->j ? 1 : 0);",
     "return (x->j > y->j) ? -1 : (x->j < y->j ? 1 : 0);"),
    ("page-table start dropped", "int64_t col = pt_start + idx / page_size;",
     "int64_t col = idx / page_size;"),
    ("offset uses quotient", "int64_t phys = page * page_size + idx % page_size;",
     "int64_t phys = page * page_size + idx / page_size;"),
    ("pad value -inf", "uint32_t u = 0xFF7FFFFFu;", "uint32_t u = 0xFF800000u;"),
    ("page_size=1 start default", "(page_size == 1 ? rs : 0)", "0"),
    ("fp16 subnormal scale", "ldexp((double)fr, -24)", "ldexp((double)fr, -22)"),
    ("bf16 shift", "(uint32_t)h << 16", "(uint32_t)h << 15"),
    ("short rows not padded", "int64_t m = n < k ? n : k;", "int64_t m = k;"),
    ("ragged offset subtracted", "int64_t v = (int64_t)raw[s] + (int64_t)offsets[r];",
     "int64_t v = (int64_t)raw[s] - (int64_t)offsets[r];"),
    ("request row dropped", "page_table[b * pt_row_stride + idx]", "page_table[idx]"),
    ("request bounds off by one", "cu_seqlens_q[q] <= r && r < cu_seqlens_q[q + 1]",
     "cu_seqlens_q[q] <= r && r <= cu_seqlens_q[q + 1]"),
    ("large ties keep the small columns", "return (x->j > y->j) ? -1 : (x->j < y->j ? 1 : 0);",
     "return (x->j < y->j) ? -1 : (x->j > y->j ? 1 : 0);"),
    ("large ties left unsorted", "        qsort(items, (size_t)m, sizeof(item_t), by_value_desc_index_asc);\n", ""),
    ("window not clamped to the width", "return len < room ? len : room;", "return len;"),
    ("start outside the width not empty", "if (row_start < 0 || row_start > width || len <= 0)",
     "if (len <= 0)"),
    ("page column outside the table kept", "if (col < 0 || col >= pt_cols) {", "if (0) {"),
]


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, label, old, new):
    src = open(ORACLE_SRC).read()
    control = not old
    assert control or src.count(old) == 1, label
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src if control else src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-w", "-o",
                           str(so), str(mutant), "-lm"])
    # run in a child process: a mutant may crash, which also counts as caught
    script = ("import sys, ctypes; sys.path[:0] = [%r, %r]; import test_oracle_pins as t; "
              "f = t.golden_failures(t._bind(ctypes.CDLL(%r))); print(len(f)); "
              "sys.exit(3 if f else 0)") % (os.path.dirname(__file__),
                                           os.path.dirname(os.path.dirname(__file__)), str(so))
    rc = subprocess.run([sys.executable, "-c", script], capture_output=True).returncode
    if control:
        assert rc == 0, "the unmodified oracle must pass every pin in the child process"
    else:
        assert rc != 0, f"mutant '{label}' passed every pin"


def test_epilogue_variants_brute_force(oracle_mod):
    """The ragged-offset and request page-table epilogues against pure Python
    (selection by sorted() on (-value, column), then the transform)."""
    rnd = random.Random(11)
    R, W, k = 9, 12, 5
    vals = [[float(rnd.choice([-2, -1, 0, 1, 1, 2, 3, 5])) for _ in range(W)] for _ in range(R)]
    scores = torch.tensor(vals, dtype=torch.float32)
    lengths = [rnd.randint(0, W) for _ in range(R)]
    starts = [rnd.randint(0, W - L) for L in lengths]
    offsets = [rnd.randint(-50, 5000) for _ in range(R)]
    cu = [0, 3, 3, 7]                       # rows 7, 8 belong to no request
    pt = [[rnd.randint(0, 999) for _ in range(10)] for _ in range(3)]

    def local_topk(r):
        row = vals[r][starts[r]:starts[r] + lengths[r]]
        return _brute(row, len(row), k)
    out = oracle_mod.ragged_offset_transform(
        scores, torch.tensor(lengths), torch.tensor(offsets), k, torch.tensor(starts))
    for r in range(R):
        assert out[r].tolist() == [i + offsets[r] if i >= 0 else -1 for i in local_topk(r)]
    out2 = oracle_mod.seqs_page_table_transform(
        scores, torch.tensor(lengths), torch.tensor(pt, dtype=torch.int32), torch.tensor(cu), k,
        torch.tensor(starts))
    for r in range(R):
        b = next((q for q in range(len(cu) - 1) if cu[q] <= r < cu[q + 1]), None)
        want = [-1] * k if b is None else [pt[b][i] if 0 <= i < 10 else -1 for i in local_topk(r)]
        assert out2[r].tolist() == want


def test_large_ties_brute_force(oracle_mod):
    """LARGE tie mode against pure Python on small alphabets (many ties)."""
    rnd = random.Random(12)
    for trial in range(200):
        n = rnd.randint(0, 20)
        k = rnd.randint(1, 24)
        vals = [float(rnd.choice([-1, 0, 0, 1, 2, 2])) for _ in range(max(n, 1))]
        row = torch.tensor(vals, dtype=torch.float32).view(1, -1)
        idx, _ = oracle_mod.topk_varlen_ties(row, torch.tensor([n], dtype=torch.int32), k, True)
        keep = sorted(range(n), key=lambda j: (-vals[j], -j))[:k]
        want = sorted(keep, key=lambda j: (-vals[j], j)) + [-1] * (k - min(k, n))
        assert idx[0].tolist() == want, (vals[:n], k)


@pytest.mark.parametrize("k", [4096, 16384])
def test_large_k_brute_force(oracle_mod, k):
    """top_k beyond 2048 (up to 16384): the oracle's selection, the SMALL and
    LARGE tie modes and the padding against pure Python sorts of rows with
    heavy ties, rows longer and shorter than k."""
    rnd = random.Random(k)
    for n in (k - 1, k, k + 1, 20000):
        vals = [float(rnd.randint(-40, 40)) / 8 for _ in range(n)]
        row = torch.tensor(vals, dtype=torch.float32)
        idx, _ = oracle_mod.select_row(row, n, k)
        assert idx.tolist() == _brute(vals, n, k), (k, n)
        small, _ = oracle_mod.topk_varlen_ties(row.view(1, -1), torch.tensor([n], dtype=torch.int32),
                                               k, False)
        assert small[0].tolist() == _brute(vals, n, k), (k, n)
        large, _ = oracle_mod.topk_varlen_ties(row.view(1, -1), torch.tensor([n], dtype=torch.int32),
                                               k, True)
        keep = sorted(range(n), key=lambda j: (-vals[j], -j))[:k]
        want = sorted(keep, key=lambda j: (-vals[j], j)) + [-1] * (k - min(k, n))
        assert large[0].tolist() == want, (k, n)
