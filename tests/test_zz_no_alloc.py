"""The allocation-free entry point (gbtopk_varlen_static_ws).

For callers that cannot allocate device memory where they need top-K (during
CUDA graph capture, under an external allocator that forbids side
allocations, inside plugin hosts), the library offers a variant that uses a
16 MiB scratch buffer compiled into the library instead of a caller
workspace.  These tests call it through the C ABI and check that, on two
calls in a row sharing that buffer, it returns what gbtopk_varlen returns
with a caller-owned workspace (bit-identical in deterministic mode, the same
tie-aware selection otherwise) and that both agree with the CPU oracle.
This file is collected last on purpose.
"""
import pytest
import torch

import oracle
import sparse_attention_top_gb300 as gb
import workloads
from parity import check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gb.load_library()
    return torch.device("cuda:0")


def _reference(c, dev, det):
    R, W = c.logits.shape
    out = torch.empty(R, c.top_k, dtype=torch.int32, device=dev)
    val = torch.empty(R, c.top_k, dtype=c.logits.dtype, device=dev)
    ws = torch.zeros(gb.gbtopk_workspace_bytes(R, W, c.top_k, c.logits.dtype),
                     dtype=torch.uint8, device=dev)
    hint = c.pre_idx.to(dev) if c.pre_idx is not None else None
    gb.gbtopk_varlen(c.logits.to(dev), c.seq_lens.to(dev), c.top_k, hint, c.next_n,
                     c.compress_ratio, out, val, det, ws)
    torch.cuda.synchronize(dev)
    return out.cpu(), val.cpu()


@pytest.mark.parametrize("case", ["decode", "tiny", "mtp_small"])
def test_static_scratch_matches_caller_workspace(dev, case):
    if case == "decode":   # 64 x 163840 fp32, top_k 2048 (about 6.3 MiB of scratch)
        c = workloads.dsv32_decode(rows=64, width=163840, top_k=2048, seed=2500)
    elif case == "tiny":
        c = workloads.tiny()
    else:
        c = workloads.dsv4_mtp(requests=8, width=40000, top_k=512, seed=4500)
    R, W = c.logits.shape
    assert gb.gbtopk_workspace_bytes(R, W, c.top_k, c.logits.dtype) <= 16 << 20
    x = c.logits.to(dev)
    seq = c.seq_lens.to(dev)
    hint = c.pre_idx.to(dev) if c.pre_idx is not None else None
    n = oracle.row_lengths(c.seq_lens.tolist(), R, c.next_n, c.compress_ratio, W)
    orc_i, _ = oracle.topk_varlen(c.logits, c.seq_lens, c.top_k, c.next_n, c.compress_ratio,
                                  return_values=False)
    for det in (True, False):
        ref_i, ref_v = _reference(c, dev, det)
        check_rows(c.logits, n, c.top_k, ref_i, orc_i, ref_v, deterministic=det)
        for call in range(2):   # two calls in a row share the library's scratch
            out = torch.full((R, c.top_k), 7, dtype=torch.int32, device=dev)
            val = torch.zeros((R, c.top_k), dtype=c.logits.dtype, device=dev)
            st = gb.gbtopk_varlen_static_ws(x, seq, c.top_k, hint, c.next_n, c.compress_ratio,
                                            out, val, det)
            assert st == gb.OK
            torch.cuda.synchronize(dev)
            if det:
                assert torch.equal(out.cpu(), ref_i)
                assert torch.equal(val.cpu().view(torch.int16 if c.logits.element_size() == 2
                                                  else torch.int32),
                                   ref_v.view(torch.int16 if c.logits.element_size() == 2
                                              else torch.int32))
            else:
                check_rows(c.logits, n, c.top_k, out, ref_i, val)
            check_rows(c.logits, n, c.top_k, out, orc_i, val, deterministic=det)


def test_static_scratch_refuses_oversized_geometry(dev):
    # 1024 x 262144 fp32 with top_k 2048 needs far more than 16 MiB of scratch
    assert gb.gbtopk_workspace_bytes(1024, 262144, 2048, torch.float32) > 16 << 20
    lib = gb.load_library()
    dummy = torch.empty(16, dtype=torch.int32, device=dev)
    st = lib.gbtopk_varlen_static_ws(dummy.data_ptr(), 0, 1024, 262144, 262144,
                                     dummy.data_ptr(), 1, 1, 2048, None, dummy.data_ptr(), None,
                                     0, None)
    assert st == gb.EWORKSPACE
