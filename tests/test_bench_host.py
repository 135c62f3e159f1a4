"""bench.py's multi-rank logic on CPU: gloo ranks in separate processes."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    q.put((rank, bench.max_over_ranks([1.0 + rank, 10.0 - rank, float(rank)])))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0, 1.0]


def test_max_over_ranks_without_a_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 1.0]) == [3.0, 1.0]


def test_reference_arm_under_torchrun_prints_once():
    """--impl reference under torchrun with 2 ranks: rank 0 prints one JSON line,
    the other rank exits 0 without work."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=%d" % port, os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


# ------------------------------------------------- algorithmic bytes (roofline)

def _shape_case(ratio, coff, head_dim, lens, capacity=None, extra_rows=0, leading=0):
    sys.path.insert(0, ROOT)
    import csa_workloads as w
    cu, cc = w.offsets(lens, ratio, leading)
    cap = int(cc[-1]) + extra_rows if capacity is None else capacity
    return w.Case("shape", ratio, coff, head_dim, list(lens), cap, int(cu[-1]), cu, cc, None, None, None, None)


def _window_term_by_enumeration(c, rows):
    """Distinct (token, half) slots the given rows read, from the oracle's gather
    window map, as bytes of kv + score (2 bf16 per column)."""
    import numpy as np
    from oracle import gather
    token, half, _, valid, real = gather.window_index(c.cu_seqlens, c.cu_seqlens_comp, c.ratio, c.coff,
                                                      c.capacity)
    sel = valid & (real if rows == "real" else np.ones_like(real))[:, None]
    h = np.broadcast_to(half[None, :], token.shape)
    return len(np.unique(token[sel] * 2 + h[sel])) * c.head_dim * 4


def _check_bytes(c):
    sys.path.insert(0, ROOT)
    import bench
    fwd, bwd = bench.algorithmic_bytes(c)
    C = c.coff * c.head_dim
    ape = 4 * c.ratio * C
    assert fwd == _window_term_by_enumeration(c, "all") + ape + 2 * c.capacity * c.head_dim
    assert bwd == (_window_term_by_enumeration(c, "real") + 2 * c.n_real_rows * c.head_dim + ape
                   + 4 * c.n_tokens * C + ape)


def test_algorithmic_bytes_of_every_workload_match_the_window_map():
    """The roofline's numerator: each consumed kv / score slot once (forward: every
    row, padding rows included; backward: real rows), counted against a brute-force
    enumeration of the oracle's window map on the benchmark layouts."""
    sys.path.insert(0, ROOT)
    import csa_workloads as w
    for name, spec in w.SPECS.items():
        kw = spec(0)
        c = _shape_case(kw["ratio"], kw["coff"], kw["head_dim"], kw["seqlens"], capacity=kw.get("capacity"),
                        extra_rows=kw.get("extra_rows", 0))
        _check_bytes(c)


def test_algorithmic_bytes_on_ragged_layouts():
    """Short and empty segments, tails, leading tokens and padding rows whose tokens
    [0, ratio) no real row reads."""
    import numpy as np
    rng = np.random.default_rng(0)
    n = 0
    while n < 400:
        ratio = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        lens = [int(x) for x in rng.integers(0, 4 * ratio + 2, int(rng.integers(1, 5)))]
        c = _shape_case(ratio, int(rng.integers(1, 3)), 8, lens, extra_rows=int(rng.choice([0, 1, 3])),
                        leading=int(rng.choice([0, 0, 2])))
        if c.capacity == 0 or c.n_tokens < ratio:
            continue
        _check_bytes(c)
        n += 1
