"""Host logic of the N > 1 benchmark path (independent replicas, no
collective in the step): the slowest rank's time is what every rank reports,
and throughput counts all replicas.  Two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is slower
        got = bench.max_over_ranks(ms, world, torch.device("cpu"))
        out[rank] = (got, bench.replica_throughput(1_000_000, world, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_slowest_time_and_total_throughput():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, tput = res[0]
    assert ms == 15.0
    assert tput == pytest.approx(2 * 1_000_000 / 0.015)


def test_launcher_starts_n_ranks_with_gloo(capfd):
    """bench.launch_ranks runs a script as N ranks under torch.distributed.run
    (the path `bench.py --gpus N` takes when started without torchrun); the
    probe rank reports the world size and the slowest rank's time."""
    import json
    import sys
    probe = os.path.join(os.path.dirname(os.path.abspath(__file__)), "bench_rank_probe.py")
    rc = bench.launch_ranks(2, probe, [])
    assert rc == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, lines
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2
    assert rec["ms_per_step"] == 11.0
    assert rec["value"] == pytest.approx(2 * 1_000_000 / 0.011)
    assert sys.executable == bench.torchrun_cmd(2, probe, [], 1)[0]


def test_bench_main_relaunches_for_gpus_n(monkeypatch):
    """`bench.py --gpus 3` without WORLD_SIZE re-executes itself as 3 ranks and
    exits with the launcher's status; under torchrun a WORLD_SIZE that differs
    from --gpus is an error."""
    calls = []
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench, "launch_ranks", lambda n, script, argv: calls.append((n, script, list(argv))) or 7)
    monkeypatch.setattr("sys.argv", ["bench.py", "--gpus", "3", "--steps", "4"])
    with pytest.raises(SystemExit) as ex:
        bench.main()
    assert ex.value.code == 7
    assert calls == [(3, os.path.abspath(bench.__file__), ["--gpus", "3", "--steps", "4"])]
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--gpus", "4"])
    with pytest.raises(SystemExit) as ex:
        bench.main()
    assert ex.value.code == 2


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.replica_throughput(8_030_261_248, 1, 20.0) == pytest.approx(8_030_261_248 / 0.02)


# ---- row-sharded step: the exchange protocol on gloo ranks -----------------
# The library's row-sharded step (adafactor_shard_begin / middle / end)
# exchanges, per tensor, the column sums of g^2, the sum of the updated row
# statistic per slice and sum(p^2) (exchange round 1), then sum(u^2) (exchange round 2).  Here
# two gloo ranks run that protocol in float64 numpy on their row blocks, with
# real all-reduces between the phases, and must reproduce the oracle on the
# whole tensors; every rank also checks that the library's exchange buffer
# sizes do not depend on its row count.
SHARD_SHAPES = [(7, 5), (2, 6, 3), (9,)]


def _shard_rows(n, world, rank):
    cuts = [0, (n * 2) // 5, n] if world == 2 else [0, n]
    return cuts[rank], cuts[rank + 1]


def _shard_worker(rank, world, port, out):
    import numpy as np

    import oracle
    from memory_efficient_optimizer_gb300 import binding as B
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        def allreduce(x):
            t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
            dist.all_reduce(t)
            return t.numpy()

        # Exchange sizes from the library (host-only query), with this rank's rows.
        n = len(SHARD_SHAPES)
        T, S = (B.adaf_tensor * n)(), (B.adaf_shard * n)()
        for k, s in enumerate(SHARD_SHAPES):
            r0, r1 = _shard_rows(s[-2] if len(s) >= 2 else s[0], world, rank)
            local = list(s)
            local[-2 if len(s) >= 2 else 0] = r1 - r0
            T[k].param = T[k].grad = 0x1000
            T[k].grad_dtype, T[k].ndim = B.ADAF_FLOAT32, len(s)
            for d, v in enumerate(local):
                T[k].shape[d] = v
            S[k].global_rows = s[-2] if len(s) >= 2 else s[0]
        _, r1b, r2b = B.adafactor_shard_sizes(T, S, n)
        sizes = torch.tensor([r1b, r2b], dtype=torch.int64)
        all_sizes = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(all_sizes, sizes)

        hp = oracle.HParams(beta1=0.9, weight_decay=0.05)
        rng = np.random.default_rng(7)
        worst = 0.0
        for k, s in enumerate(SHARD_SHAPES):
            full_p = rng.normal(0, 0.3, s)
            gs = [rng.normal(0, 0.01, s) for _ in range(3)]
            ref = full_p.copy()
            rst = oracle.State(s, beta1=True)
            fact = len(s) >= 2
            H = s[-2] if fact else s[0]
            r0, r1 = _shard_rows(H, world, rank)
            sl = (Ellipsis, slice(r0, r1), slice(None)) if fact else (slice(r0, r1),)
            p = full_p[sl].copy()
            lead = int(np.prod(s[:-2])) if fact else 1
            W = s[-1] if fact else 1
            N = full_p.size
            row = np.zeros(p.shape[:-1]) if fact else None
            col = np.zeros(s[:-2] + (W,)) if fact else None
            v = None if fact else np.zeros(p.shape)
            m1 = np.zeros(p.shape)
            for t, gfull in enumerate(gs, start=1):
                oracle.step(ref, gfull, rst, t, hp)
                g = gfull[sl]
                rho = min(1e-2, 1 / np.sqrt(t))
                b2 = 1 - t ** hp.decay_rate
                q = g * g + hp.eps[0]
                # begin: local statistics
                if fact:
                    row = b2 * row + (1 - b2) * q.mean(axis=-1)
                    x1 = np.concatenate([q.sum(axis=-2).ravel(), row.reshape(lead, -1).sum(axis=-1),
                                         [np.sum(p * p)]])
                else:
                    v = b2 * v + (1 - b2) * q
                    x1 = np.array([np.sum(p * p)])
                x1 = allreduce(x1)  # exchange round 1
                # middle: column statistic, mean(row), alpha; local sum(u^2)
                psq = x1[-1]
                alpha = rho * max(hp.eps[1], np.sqrt(psq / N))
                if fact:
                    csum = x1[:lead * W].reshape(col.shape)
                    col = b2 * col + (1 - b2) * csum / H
                    mrow = x1[lead * W:lead * W + lead].reshape(s[:-2] + (1,)) / H
                    u = g / np.sqrt(row[..., None] / mrow[..., None] * col[..., None, :])
                else:
                    u = g / np.sqrt(v)
                x2 = allreduce(np.array([np.sum(u * u)]))  # exchange round 2
                # end: clip, beta1, weight decay, update
                u = alpha * u / max(1.0, np.sqrt(x2[0] / N) / hp.clip_threshold)
                m1 = hp.beta1 * m1 + (1 - hp.beta1) * u
                p = p - hp.weight_decay * alpha * p - m1
            err = np.max(np.abs(p - ref[sl]) / np.maximum(np.abs(ref[sl]), 1e-12))
            worst = max(worst, float(err))
            if fact:
                worst = max(worst, float(np.max(np.abs(col.ravel() - rst.col.ravel()) / rst.col.ravel())))
        out[rank] = (worst, [tuple(x.tolist()) for x in all_sizes])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_row_sharded_exchange_protocol_on_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_shard_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        worst, sizes = res[rank]
        assert worst < 1e-12, (rank, worst)
        assert len(set(sizes)) == 1, sizes  # exchange sizes agree across ranks
