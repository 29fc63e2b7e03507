"""The benchmark's data-parallel chain step on NCCL (one rank on one GPU, in a
spawned process): the valid-count all-reduce, the linear CE in sum mode scaled
by 1 / n_valid, and the loss, dW and dw all-reduces give the plain step's
gradients and its mean loss.  The exchanges across several ranks are covered on
gloo (tests/test_bench_host.py, tests/test_data_parallel_recipe.py)."""
import os
import socket
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _child(port, q):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": "0", "WORLD_SIZE": "1",
                       "NCCL_NVLS_ENABLE": "0"})
    try:
        import torch
        import torch.distributed as dist
        import transformer_rmsnorm_fwd_gb300 as L
        import bench
        L.load()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        dist.init_process_group("nccl", rank=0, world_size=1)
        inputs = bench.gen_inputs(1024)
        plain = bench.Chain(L, inputs, dev)
        plain.step()
        n = int((inputs["labels"] != -100).sum())
        dp = bench.DataParallel(dist, n, dev)
        chain = bench.Chain(L, inputs, dev, dp)
        chain.step()
        torch.cuda.synchronize()

        def rel(a, b):
            return float((a.float() - b.float()).abs().max() / b.float().abs().max())

        out = (float(plain.loss.item()), dp.mean_loss(float(chain.loss.item())), rel(chain.dW, plain.dW),
               rel(chain.dw, plain.dw), rel(chain.dX, plain.dX))
        dist.destroy_process_group()
        q.put(("ok", out))
    except Exception as e:   # reported to the test
        q.put(("error", repr(e)))


def test_data_parallel_step_on_one_nccl_rank(cuda_lib):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_child, args=(_free_port(), q))
    p.start()
    status, out = q.get(timeout=600)
    p.join(timeout=120)
    assert status == "ok", out
    assert p.exitcode == 0
    lp, ld, rdW, rdw, rdX = out
    assert abs(lp - ld) <= 1e-5 * abs(lp)
    # one rank: the all-reduces are identities, and sum mode with 1 / n_valid reproduces the
    # mean's gradients within rounding of the scale
    assert rdW <= 1e-2 and rdw <= 1e-2 and rdX <= 1e-2
