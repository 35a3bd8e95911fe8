"""The N > 1 bench path on the host: replicas, one process per GPU, no data-path collective.

Each rank runs its own copy of the whole hot path on its own GPU; the only collectives are the
barrier around the timed region and the max of the per-rank times. These tests run that plumbing
as two `gloo` ranks on the CPU: the rendezvous, the barrier, the max over ranks, and that two
replicas of the fork step's host path (match, evict, allocate, insert) make identical decisions.
"""
import hashlib
import json
import os
import socket
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _small_fork_workload():
    from synth import workloads as W
    return W.fork_mixed_step(layers=1, pool_slots=20_000, n_programs=4, prefix_len=300,
                             n_forks=3, suffix_len=40, n_decode=8, dec_lo=64, dec_hi=512,
                             free_at_start=1024, max_steps=8, filler_len=200)


def _replica_digest(steps=3):
    """One replica of the fork step's host path: cache phases, then `steps` extend steps."""
    from prefix_cached_paged_gb300.runtime import HostCache
    fm = _small_fork_workload()
    w = fm.workload
    hc = HostCache(w.pool_slots, w.max_ctx, w.pool_order)
    for ph in w.phases:
        for s in ph.seqs:
            hc.finish(hc.plan([s], match_all=True), keep_locked=ph.keep_locked)
    h = hashlib.sha256()
    evicted = 0
    for step in range(steps):
        p = hc.plan(fm.extend_seqs(step))
        for arr in (p.prefix_len, p.out_loc, p.qo_indptr, p.rows):
            h.update(np.ascontiguousarray(arr).tobytes())
        evicted += int(p.evicted)
        hc.finish(p)
    return h.hexdigest(), evicted


def _worker(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    try:
        r, w, _ = bench.dist_init()
        bench.barrier(w)
        m = bench.max_over_ranks(float(rank) + 0.5, w)
        digest, evicted = _replica_digest()
        gathered = [None] * w
        dist.all_gather_object(gathered, (digest, evicted))
        bench.barrier(w)
        queue.put((rank, r, w, dist.get_backend(), m, gathered))
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        queue.put((rank, "error", repr(e)))
        raise


def test_two_gloo_ranks_run_identical_replicas():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = []
    try:
        for _ in range(2):
            out.append(q.get(timeout=240))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs), out
    out.sort(key=lambda t: t[0])
    for rank, (rk, r, w, backend, m, gathered) in enumerate(out):
        assert (rk, r, w, backend) == (rank, rank, 2, "gloo")
        assert m == 1.5                        # max over ranks of 0.5 and 1.5
        assert gathered[0] == gathered[1]      # identical replica decisions
        assert gathered[0][1] > 0              # the small pool forces eviction every run
    # and they equal a single-process run of the same replica
    sys.path.insert(0, ROOT)
    assert out[0][5][0] == _replica_digest()


def test_reference_arm_under_torchrun_prints_once():
    """Under torchrun rank 0 alone runs the reference arm and prints; the other rank exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-budget", "2",
           "--layers", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
