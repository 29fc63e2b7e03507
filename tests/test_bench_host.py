"""Host-side logic of bench.py: the multi-rank timing reduction (world size
2 over gloo on CPU), the algorithmic work per call, and the JSON contract of
the reference (oracle) arm on a tiny sequence."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world)})
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mx = bench.max_over_ranks(10.0 + rank, dist)
    sm = bench.sum_over_ranks(100.0 * (rank + 1), dist)
    q.put((rank, mx, sm))
    dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 11.0, 300.0), (1, 11.0, 300.0)]


def test_single_process_reduction_is_identity():
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.sum_over_ranks(7.0, None) == 7.0


def test_algorithmic_work():
    a = bench.algorithmic(8192)
    assert a["swiglu_fwd"] == 3 * 8192 * 11008 * 2            # 541 MB, the [4,2048,11008] SwiGLU forward
    assert a["swiglu_bwd"] == 5 * 8192 * 11008 * 2
    assert a["rope_fwd"] == 2 * 2 * 8192 * 32 * 128 * 2
    assert a["linear_ce_flops"] == 6 * 8192 * 4096 * 151936


@pytest.mark.slow
def test_reference_arm_json_contract():
    env = dict(os.environ)
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--seq", "256"], capture_output=True, text=True, env=env, timeout=600)
    assert p.returncode == 0, p.stderr
    d = json.loads(p.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_launch_count_per_step():
    """The benchmark's gpu_launches claim: 39 launches of this library per chain step
    at seq 32768 (the ncu launch list of the step, profiles/launches_qwen_chain_s32768.md,
    counts 117 over 3 steps): RMSNorm, RoPE and SwiGLU forwards, the linear CE (label
    scan, sort and starts, 4 chunks x (2 logits launches, dlogits, 3 dX slab launches,
    dW), loss reduction), SwiGLU and RoPE backwards, RMSNorm backward (2)."""
    class _C:
        S = 32768
    assert bench.Chain.launches_per_step(_C()) == 39
    with open(os.path.join(ROOT, "profiles", "launches_qwen_chain_s32768.md")) as f:
        text = f.read()
    assert "-c 117" in text and "TOTAL" in text
    total = [l for l in text.splitlines() if l.startswith("TOTAL")][0].split()
    assert int(total[1]) == 3 * 39
