"""Two-rank CPU (gloo) checks of the multi-process path of bench.py.

Rows are independent, so N GPUs run N replicas on their own batches (weak
scaling) and only the timing and row totals cross ranks.  These tests launch
two processes with torch.distributed.run on 127.0.0.1 and no GPU.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout=240, **extra_env):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1", **extra_env)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def _json_lines(text):
    out = []
    for line in text.splitlines():
        line = line.strip()
        if line.startswith("{"):
            out.append(json.loads(line))
    return out


def test_two_rank_reductions_and_batches(tmp_path):
    r = _torchrun([os.path.join("tests", "dist_worker.py")], GBTOPK_DIST_OUT=str(tmp_path))
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    lines = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    assert [l["rank"] for l in lines] == [0, 1]
    assert all(l["ok"] and l["world"] == 2 for l in lines)


def test_reference_arm_prints_once_on_rank0():
    # the CPU oracle arm under two ranks: rank 0 alone times and prints
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                   "--warmup", "0"])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_gpus_flag_starts_its_own_ranks():
    """`bench.py --gpus 2` started without a launcher runs two ranks itself
    (through torch.distributed.run); the reference arm then prints one line
    from rank 0 with n_gpus 2."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    for key in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(key, None)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def test_gpus_flag_must_match_the_launcher():
    """Under a launcher, --gpus must equal WORLD_SIZE (no silent n_gpus 1)."""
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "4", "--steps", "1",
                   "--warmup", "0"])
    assert r.returncode != 0 and "WORLD_SIZE" in (r.stdout + r.stderr)
