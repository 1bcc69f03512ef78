"""The multi-rank path of bench.py on CPU: world_size 2 over gloo (127.0.0.1).
Every rank runs an independent replica; rank 0 reports the slowest rank's time
and all ranks' tokens. The reference arm runs on rank 0 only."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 100.0 + 50.0 * rank          # rank 1 is the slower replica
    worst = bench.max_over_ranks(ms, world, "cpu")
    out[rank] = (worst, bench.job_tokens_per_s(world, 16384, 10, worst), bench.dist_env())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_over_gloo():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        worst, tps, env = out[r]
        assert worst == 150.0
        assert tps == pytest.approx(2 * 16384 * 10 / 0.150)
        assert env == (r, world, r)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(42.0, 1, "cpu") == 42.0
    assert bench.job_tokens_per_s(1, 1000, 4, 2000.0) == pytest.approx(2000.0)


def test_reference_arm_is_rank0_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), dict(gpus=2, steps=1, warmup=0))()
    bench.run_reference(args, None, 1024)   # returns at once on rank 1, prints nothing
    assert capsys.readouterr().out == ""


def test_bench_defines_every_path_it_dispatches():
    """bench.py's entry points all exist (a missing one would only surface on a
    GPU run)."""
    import ast
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py")).read()
    tree = ast.parse(src)
    defined = set()
    for n in ast.walk(tree):
        if isinstance(n, (ast.FunctionDef, ast.ClassDef)):
            defined.add(n.name)
        elif isinstance(n, (ast.Import, ast.ImportFrom)):
            defined.update((a.asname or a.name).split(".")[0] for a in n.names)
        elif isinstance(n, ast.Name) and isinstance(n.ctx, ast.Store):
            defined.add(n.id)
        elif isinstance(n, ast.arg):
            defined.add(n.arg)
    called = {n.func.id for n in ast.walk(tree)
              if isinstance(n, ast.Call) and isinstance(n.func, ast.Name)}
    builtins = set(dir(__import__("builtins")))
    missing = {c for c in called if c not in defined and c not in builtins}
    assert not missing, missing


# ---------------------------------------------------------------- token-sharded loss

def _oracle_fwd_bwd(H, W, y, chunk, ignore_index, compute_dW, n_valid_total):
    """Stand-in for the library's fused call with a given normaliser on the CPU
    (this test checks the exchange around it; the call itself is parity-tested on
    the GPU): the rank's loss sum and G scaled by 1 / n_valid_total."""
    from oracle import lce_oracle as O
    n = int(n_valid_total.reshape(-1)[0])
    r = O.forward_backward(H, W, y, dloss=1.0 / n if n else 0.0, reduction="sum",
                           ignore_index=ignore_index)
    dW = torch.from_numpy(r["dW"]).to(torch.float32) if compute_dW else None
    loss = r["loss"] / n if n else 0.0
    return (torch.tensor([loss], dtype=torch.float32), torch.from_numpy(r["lse"]).float(),
            torch.from_numpy(r["dH"]).float(), dW)


def _oracle_count(y, V, ignore_index):
    """Stand-in for the library's valid-row count (the oracle's reading)."""
    from oracle import lce_oracle as O
    valid, _ = O.valid_rows(y, V, ignore_index)
    return torch.tensor([int(valid.sum())], dtype=torch.int64)


def _sharded_worker(rank, world, port, out, cuts, compute_dW):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from lce_synth import make_inputs
    from linear_cross_entropy_chunked_gb300.sharded import sharded_fwd_bwd
    H, W, y = make_inputs(96, 16, 40, seed=7, n_ignored=9)
    y[5] = 40                        # out of range: counts as ignored
    lo, hi = cuts[rank], cuts[rank + 1]
    loss, lse, dH, dW = sharded_fwd_bwd(H[lo:hi], W, y[lo:hi], compute_dW=compute_dW,
                                        fwd_bwd=_oracle_fwd_bwd, count=_oracle_count)
    out[rank] = (float(loss), dH.numpy(), None if dW is None else dW.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("cuts,compute_dW", [((0, 40, 96), True), ((0, 0, 96), True),
                                             ((0, 70, 96), False)])
def test_token_sharded_loss_equals_the_whole_batch(cuts, compute_dW):
    """Two ranks over gloo, each with a slice of the rows (one may be empty):
    the global loss and dW on every rank, and each rank's dH rows, equal the
    oracle's on the whole batch."""
    from lce_synth import make_inputs
    from oracle import lce_oracle as O
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_sharded_worker, args=(world, port, out, cuts, compute_dW), nprocs=world, join=True)
    H, W, y = make_inputs(96, 16, 40, seed=7, n_ignored=9)
    y[5] = 40
    ref = O.forward_backward(H, W, y)
    dH = np.concatenate([out[r][1] for r in range(world)])
    for r in range(world):
        assert out[r][0] == pytest.approx(ref["loss"], rel=1e-6)
        if compute_dW:
            assert np.allclose(out[r][2], ref["dW"], rtol=1e-5, atol=1e-7)
        else:
            assert out[r][2] is None
    assert np.allclose(dH, ref["dH"], rtol=1e-5, atol=1e-7)
