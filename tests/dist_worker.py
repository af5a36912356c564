"""One rank of the two-process CPU check of bench.py's multi-process plumbing.

Launched by tests/test_dist_gloo.py under torch.distributed.run with the gloo
backend (no GPU): it exercises the rank/world discovery, the barrier, the
max-over-ranks time and sum-over-ranks row reductions that bench.py uses to
form its whole-job number, and checks that every rank draws its own batch
(weak scaling: rows are independent, no collective on the data path).
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    rank, world, local = bench.dist_init(2)
    assert dist.is_initialized() and dist.get_backend() == "gloo"
    assert world == 2 and rank in (0, 1) and local == rank
    # the whole-job number: rows of all ranks over the slowest rank's time
    ms = [12.5, 20.0][rank]
    rows = [64, 64][rank]
    assert bench.reduce_max(ms) == 20.0
    assert bench.reduce_sum(float(rows)) == 128.0
    bench.barrier()
    # each rank's batch is seeded by its rank, so the ranks' inputs differ
    case = bench._varlen_case("dsv32_decode", rank)
    assert tuple(case.logits.shape) == (64, 163840) and case.top_k == 2048
    sig = float(case.logits[:, :256].double().sum())
    sigs = [None, None]
    dist.all_gather_object(sigs, sig)
    assert sigs[0] != sigs[1], "ranks drew the same batch"
    bench.barrier()
    # one result file per rank (the ranks share stdout, where lines can interleave)
    with open(os.path.join(os.environ["GBTOPK_DIST_OUT"], f"rank{rank}.json"), "w") as f:
        json.dump({"rank": rank, "world": world, "ok": True}, f)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
