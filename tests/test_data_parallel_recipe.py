"""Token-sharded (data-parallel) use of the operators, two gloo ranks on CPU.

The rows of every operator are independent, so a batch split over ranks needs
only the exchanges that the mean and the weight gradients imply:
  - linear cross-entropy: the number of valid (not ignored) tokens summed over
    ranks before the logit gradient is scaled, then the loss and dW summed;
    each rank calls the operator in sum mode with grad_scale = 1 / n_valid of
    the whole batch, which the C-ABI's reduction / grad_scale arguments allow;
  - RMSNorm: dw summed over ranks (dx stays local).
Each rank runs the fp64 oracle on its shard; rank 0 checks the exchanged
results against the oracle on the unsharded batch (mean reduction).  The
GPU side of the same composition (two shard calls through the C-ABI) is
test_linear_ce_token_shards_compose_to_mean in test_gpu_linear_ce.py."""
import os
import socket
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

T, H, V, WORLD = 48, 16, 40, 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _problem():
    import datagen
    X = datagen.normal(71, "dpX", (T, H), "f32")
    W = datagen.normal(71, "dpW", (V, H), "f32", 0.0, 0.3)
    lab = datagen.labels(71, "dpl", T, V, 0.2)
    lab[3] = lab[5] = lab[7] = -100          # rank 0 holds more ignored rows than rank 1
    dy = datagen.normal(71, "dpdy", (T, H), "f32")
    xr = datagen.normal(71, "dpx", (T, H), "f32")
    w = datagen.normal(71, "dpw", (H,), "f32", 1.0, 0.1)
    return X, W, lab, dy, xr, w


def _rank(rank, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(WORLD)})
    import torch
    import torch.distributed as dist
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        X, W, lab, dy, xr, w = _problem()
        sl = slice(rank * T // WORLD, (rank + 1) * T // WORLD)
        # linear CE: exchange n_valid first, then scale by the global count
        n = torch.tensor([int((lab[sl] != -100).sum())], dtype=torch.int64)
        dist.all_reduce(n)
        n_global = int(n.item())
        o = oracle.linear_ce(X[sl], W, lab[sl], reduction="sum", grad_scale=1.0 / n_global)
        loss = torch.tensor([o["loss"]], dtype=torch.float64)
        dW = torch.from_numpy(o["dW"].copy())
        dist.all_reduce(loss)
        dist.all_reduce(dW)
        # RMSNorm backward: dw summed over ranks
        dx, dw = oracle.rmsnorm_bwd(dy[sl], xr[sl], w, 1e-6)
        dwt = torch.from_numpy(dw.copy())
        dist.all_reduce(dwt)
        dXs = [torch.zeros(T // WORLD, H, dtype=torch.float64) for _ in range(WORLD)]
        dist.all_gather(dXs, torch.from_numpy(o["dX"].copy()))
        dxs = [torch.zeros(T // WORLD, H, dtype=torch.float64) for _ in range(WORLD)]
        dist.all_gather(dxs, torch.from_numpy(dx.copy()))
        if rank == 0:
            q.put({"loss": loss.item() / n_global, "dW": dW.numpy(), "dX": torch.cat(dXs).numpy(),
                   "dw": dwt.numpy(), "dx": torch.cat(dxs).numpy(), "n": n_global})
    finally:
        dist.destroy_process_group()


def test_token_sharded_linear_ce_and_rmsnorm_match_the_unsharded_batch():
    import torch.multiprocessing as mp
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(WORLD)]
    for p in ps:
        p.start()
    got = q.get(timeout=180)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    X, W, lab, dy, xr, w = _problem()
    full = oracle.linear_ce(X, W, lab)
    assert got["n"] == int((lab != -100).sum())
    assert abs(got["loss"] - full["loss"]) <= 1e-12 * abs(full["loss"])
    assert np.max(np.abs(got["dW"] - full["dW"])) <= 1e-12 * np.max(np.abs(full["dW"]))
    assert np.max(np.abs(got["dX"] - full["dX"])) <= 1e-12 * np.max(np.abs(full["dX"]))
    dx, dw = oracle.rmsnorm_bwd(dy, xr, w, 1e-6)
    assert np.max(np.abs(got["dw"] - dw)) <= 1e-12 * np.max(np.abs(dw))
    assert np.array_equal(got["dx"], dx)


def test_per_rank_mean_is_not_the_batch_mean():
    """The exchange is needed: averaging each shard's own mean loss differs from
    the batch mean when the shards hold different numbers of ignored tokens."""
    import oracle
    X, W, lab, _, _, _ = _problem()
    h = T // WORLD
    per = [oracle.linear_ce(X[i * h:(i + 1) * h], W, lab[i * h:(i + 1) * h])["loss"] for i in range(WORLD)]
    assert abs(np.mean(per) - oracle.linear_ce(X, W, lab)["loss"]) > 1e-6
