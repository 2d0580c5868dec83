"""The data-parallel exchange on CPU: two gloo ranks, each with its own batch,
sum their load counts and apply the same sign update against the global mean
load, so their biases stay equal and match one rank holding both batches.
The update here is the oracle's (no GPU); the GPU layer passes the C-ABI
update through the same mixture_experts_layer_88_b300.parallel.balance_step."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import moe_oracle as O

E, K, T_LOCAL = 16, 4, 64


def _rank_T(rank):
    """Ranks hold batches of different sizes (64 and 96 tokens)."""
    return T_LOCAL + 32 * rank


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _Cfg:
    def __init__(self, T):
        self.T, self.K, self.E, self.gamma = T, K, E, 1e-3


def _rank_counts(rank):
    rng = np.random.default_rng(100 + rank)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(_rank_T(rank))])
    return np.bincount(idx.reshape(-1), minlength=E).astype(np.int32)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from mixture_experts_layer_88_b300 import parallel
    counts = torch.from_numpy(_rank_counts(rank))
    bias = torch.full((E,), 0.25, dtype=torch.float32)
    seen = {}

    def update(cfg, c, b):
        seen["T"] = cfg.T
        nb, _ = O.update_bias(c.numpy(), b.numpy(), cfg.T, cfg.K, cfg.gamma)
        b.copy_(torch.from_numpy(nb))
        return b

    parallel.balance_step(_Cfg(_rank_T(rank)), counts, bias, update)
    out[rank] = (counts.numpy().copy(), bias.numpy().copy(), seen["T"])
    dist.destroy_process_group()


def test_two_rank_balance_step_keeps_biases_equal():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    c0, b0, t0 = res[0]
    c1, b1, t1 = res[1]
    total = _rank_counts(0) + _rank_counts(1)
    np.testing.assert_array_equal(c0, total)
    np.testing.assert_array_equal(c1, total)
    T_all = _rank_T(0) + _rank_T(1)
    assert t0 == t1 == T_all
    assert np.array_equal(b0.view(np.uint32), b1.view(np.uint32))
    # equals one process updating on the whole batch
    want, _ = O.update_bias(total, np.full(E, 0.25, np.float32), T_all, K, 1e-3)
    assert np.array_equal(b0.view(np.uint32), want.view(np.uint32))
    # and differs from what rank 0 alone would have done on its half
    alone, _ = O.update_bias(_rank_counts(0), np.full(E, 0.25, np.float32), _rank_T(0), K, 1e-3)
    assert not np.array_equal(alone, want)


def _worker_peer_dies(rank, world, port, out):
    """Rank 1 leaves between steps (before the count exchange); rank 0 must
    get an error from its all-reduce within the process group's timeout
    instead of waiting for ever."""
    import datetime
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    if rank == 1:
        os._exit(0)                       # gone without a word, between steps
    from mixture_experts_layer_88_b300 import parallel
    counts = torch.from_numpy(_rank_counts(rank))
    bias = torch.zeros((E,), dtype=torch.float32)
    t0 = time.monotonic()
    try:
        parallel.balance_step(_Cfg(T_LOCAL), counts, bias, lambda cfg, c, b: b, T_global=2 * T_LOCAL)
        out[rank] = ("no error", time.monotonic() - t0)
    except Exception as e:               # noqa: BLE001  (gloo raises RuntimeError)
        out[rank] = (type(e).__name__, time.monotonic() - t0)
    # the bias was not touched by a step that could not see the global load
    out["bias_untouched"] = bool(torch.count_nonzero(bias).item() == 0)


def test_peer_leaving_is_reported_not_waited_for():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker_peer_dies, args=(r, 2, port, out))
                 for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        alive = [p for p in procs if p.is_alive()]
        for p in alive:
            p.kill()
        assert not alive, "a rank waited for a peer that had left"
        res = dict(out)
    kind, secs = res[0]
    assert kind != "no error"
    assert secs < 60
    assert res["bias_untouched"]


# ---------------------------------------------------------------- training

TG = dict(T=5, d=8, E=8, K=2, S=1, I=4)


def _train_layer():
    rng = np.random.default_rng(21)
    E, S, d, I = TG["E"], TG["S"], TG["d"], TG["I"]
    return {"centroids": rng.normal(0, 0.5, (E, d)),
            "bias": rng.uniform(-0.05, 0.05, E).astype(np.float32),
            "w13": rng.normal(0, 0.5, (E, 2 * I, d)), "w2": rng.normal(0, 0.5, (E, d, I)),
            "ws13": rng.normal(0, 0.5, (S, 2 * I, d)), "ws2": rng.normal(0, 0.5, (S, d, I))}


def _rank_batch(rank):
    rng = np.random.default_rng(300 + rank)
    return (rng.normal(0, 1.0, (TG["T"], TG["d"])), rng.normal(0, 1.0, (TG["T"], TG["d"])))


def _worker_grads(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from mixture_experts_layer_88_b300 import parallel
    inp = _train_layer()
    x, dout = _rank_batch(rank)
    inp["x"] = x
    g = O.moe_layer_backward(inp, TG["K"], dout, 1, O.SIGMOID, 1)
    grads = {k: torch.from_numpy(np.ascontiguousarray(g[k])) for k in
             ("dx", "dcentroids", "dw13", "dw2", "dws13", "dws2")}
    parallel.allreduce_grads(grads)
    out[rank] = {k: v.numpy().copy() for k, v in grads.items()}
    dist.destroy_process_group()


def test_two_rank_gradient_allreduce_equals_whole_batch():
    """Two gloo ranks, each with the oracle's backward of its own tokens: after
    allreduce_grads every rank holds the whole batch's parameter gradients
    (the oracle on both batches at once); dx stays each rank's own."""
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker_grads, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    inp = _train_layer()
    (x0, d0), (x1, d1) = _rank_batch(0), _rank_batch(1)
    inp["x"] = np.concatenate([x0, x1])
    whole = O.moe_layer_backward(inp, TG["K"], np.concatenate([d0, d1]), 1, O.SIGMOID, 1)
    for k in ("dcentroids", "dw13", "dw2", "dws13", "dws2"):
        for r in (0, 1):
            np.testing.assert_allclose(res[r][k], whole[k], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res[0]["dx"], whole["dx"][:TG["T"]], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res[1]["dx"], whole["dx"][TG["T"]:], rtol=1e-12, atol=1e-12)
