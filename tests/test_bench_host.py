"""Host-side checks of bench.py's multi-rank plumbing (no GPU): the
max-over-ranks timing reduction on two gloo ranks, and the reference arm's
rank handling (rank 0 prints one JSON line, other ranks exit quietly)."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.0], world)
    dist.barrier()
    q.put((rank, out))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == results[1] == [2.0, 10.0, 3.0]


def _bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=env, timeout=600)


def test_reference_arm_rank0_prints_one_line():
    r = _bench({"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"}, "--impl", "reference",
               "--workload", "tiny", "--gpus", "2", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "routed tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference",
               "--workload", "tiny", "--gpus", "2", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_warmup_below_three_is_refused():
    r = _bench({}, "--impl", "reference", "--workload", "tiny", "--warmup", "2")
    assert r.returncode != 0


def test_cover_tokens_reaches_each_experts_block_edges():
    """The sampled full-size checks pick, per expert, the tokens of its first
    routed row, of its last block's first row and of its last live row."""
    import numpy as np

    from oracle import routing
    from tests.gpu_util import cover_tokens
    rng = np.random.default_rng(0)
    M, k, E = 700, 2, 4
    ids = rng.integers(0, E, size=(M, k)).astype(np.int32)
    toks = cover_tokens(ids, E, 40, 1)
    route = routing.align_permute(ids, E, 128)
    sid, offs, cnt = route["sorted_token_ids"], route["expert_offsets"], route["expert_counts"]
    for e in range(E):
        lo, c = int(offs[e]), int(cnt[e])
        for row in (lo, lo + (c - 1) // 128 * 128, lo + c - 1):
            assert sid[row] // k in toks
    assert len(toks) == 40 and np.all(np.diff(toks) > 0)
