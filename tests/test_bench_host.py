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
    b = bench.algorithmic(8192, 7373)
    assert b["linear_ce_flops"] == 6 * 7373 * 4096 * 151936 and b["linear_ce_flops_all_tokens"] == a["linear_ce_flops"]


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
    """The benchmark's gpu_launches claim per chain step at seq 32768: RMSNorm, RoPE and
    SwiGLU forwards, the linear CE (label scan, sort and starts, 4 chunks x (2 logits
    launches, dlogits, 3 dX slab launches, dW), loss reduction, and with ignored labels
    the 6 launches that compact the other tokens and put the results back), SwiGLU and
    RoPE backwards, RMSNorm backward (2): 39 with every label valid (an ncu launch list
    of 3 such steps counted 117), 45 with the chain's 10 % ignored (29491 valid tokens:
    chunks of 8192, 8192, 8192 and 4915 rows)."""
    class _C:
        S = 32768
    assert bench.Chain.launches_per_step(_C()) == 39
    assert 3 * bench.Chain.launches_per_step(_C()) == 117

    class _D:
        S, n_valid = 32768, 29491
    assert bench.Chain.launches_per_step(_D()) == 45


def test_cpu_model_names_x86_and_arm_hosts():
    assert bench.cpu_model("processor\t: 0\nmodel name\t: Intel(R) Xeon(R) Platinum 8480C\n") == \
        "Intel(R) Xeon(R) Platinum 8480C"
    arm = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n"
    assert bench.cpu_model(arm) == "Arm Neoverse V2 (implementer 0x41, part 0xd4f)"
    assert bench.cpu_model(arm, "Architecture: aarch64\nModel name: Neoverse-V2\n") == "Neoverse-V2"
    assert bench.cpu_model("processor\t: 0\nCPU implementer\t: 0x61\nCPU part\t: 0x001\n") == \
        "Arm implementer 0x61, part 0x001"


class _RecordingLib:
    """Stands in for the CUDA library: records the order of the operator calls."""
    LIGER_BF16 = 1

    def __init__(self, log):
        self.log = log

    def liger_rmsnorm_bwd_workspace(self, rows, cols):
        return 16

    def liger_linear_ce_workspace(self, T, H, V, chunk, dtype):
        return 16

    def __getattr__(self, name):
        if not name.startswith("liger_"):
            raise AttributeError(name)

        def call(*args, **kw):
            self.log.append((name, kw.get("reduction", None), kw.get("grad_scale", None)))
        return call


class _RecordingDist:
    """Stands in for torch.distributed on one rank whose peer holds 30 valid labels."""

    def __init__(self, log):
        self.log = log

    def all_reduce(self, t, op=None):
        self.log.append(("all_reduce", tuple(t.shape), None))
        if t.dtype.is_floating_point is False:
            t += 30


def test_data_parallel_step_issues_the_exchanges_in_order(monkeypatch):
    """The chain step under data parallelism: the valid-label count is summed over
    ranks before the linear-CE, which runs in sum mode scaled by 1 / that count;
    after the backward the loss, dW [V, H] and the RMSNorm dw [H] are summed."""
    import numpy as np
    import torch
    monkeypatch.setattr(bench, "HIDDEN", 8)
    monkeypatch.setattr(bench, "INTER", 12)
    monkeypatch.setattr(bench, "VOCAB", 10)
    S = 4
    inputs = {k: np.zeros(sh, np.float32) for k, sh in
              {"x": (S, 8), "w": (8,), "dy_r": (S, 8), "q": (1, S, 2, 4), "k": (1, S, 2, 4), "dq": (1, S, 2, 4),
               "dk": (1, S, 2, 4), "gate": (S, 12), "up": (S, 12), "dy_s": (S, 12), "X": (S, 8),
               "W": (10, 8)}.items()}
    inputs["labels"] = np.array([1, -100, 3, 4], np.int64)
    log = []
    dp = bench.DataParallel(_RecordingDist(log), int((inputs["labels"] != -100).sum()), "cpu")
    ch = bench.Chain(_RecordingLib(log), inputs, torch.device("cpu"), dp)
    ch.step()
    names = [e[0] for e in log]
    assert names == ["liger_rmsnorm_fwd", "liger_rope_fwd", "liger_swiglu_fwd", "all_reduce",
                     "liger_linear_ce_fwd_bwd", "liger_swiglu_bwd", "liger_rope_bwd", "liger_rmsnorm_bwd",
                     "all_reduce", "all_reduce", "all_reduce"]
    assert log[3][1] == (1,)                                  # the count
    assert log[4][1:] == ("sum", 1.0 / 33)                    # 3 local + 30 on the peer
    assert [e[1] for e in log[8:]] == [(1,), (10, 8), (8,)]   # loss, dW, dw
    assert dp.mean_loss(66.0) == 2.0


def _dp_worker(rank, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": "2"})
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    dp = bench.DataParallel(dist, 5 + 2 * rank, "cpu")
    n = dp.valid_count()
    loss = torch.tensor([1.5 * (rank + 1)])
    dW = torch.full((3, 2), float(rank + 1))
    dw = torch.tensor([rank, 1.0])
    dp.reduce_grads(loss, dW, dw)
    q.put((rank, n, float(loss.item()), dW.tolist(), dw.tolist(), dp.mean_loss(float(loss.item()))))
    dist.destroy_process_group()


def test_data_parallel_exchanges_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_dp_worker, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, n, loss, dW, dw, mean in out:
        assert n == 12 and loss == 4.5 and dW == [[3.0, 3.0]] * 3 and dw == [1.0, 2.0] and mean == 4.5 / 12


def test_linear_ce_algorithmic_bytes():
    """The roofline's algorithmic bytes, counted by hand for small shapes. One chunk, no
    token ignored (T = 4, H = 8, V = 16): 10*T*V chunk-buffer bytes + W read twice + bf16
    dW + X read twice and dX written once. Two chunks with 3 of 10 tokens ignored (chunk 4,
    7 valid): the fp32 dW sum adds one write and one read, W is read twice per chunk, and
    the compaction adds the gather (7 rows read and written) and the scatter (7 rows read,
    10 written)."""
    assert bench.linear_ce_algorithmic_bytes(4, 4, 8, 16) == 10 * 4 * 16 + 2 * 16 * 8 * 2 + 16 * 8 * 2 + 3 * 4 * 8 * 2
    b = bench.linear_ce_algorithmic_bytes(7, 10, 8, 16, chunk=4)
    assert b == (10 * 7 * 16 + 4 * 16 * 8 * 2 + 2 * 16 * 8 * 4 + 16 * 8 * 2 + 3 * 7 * 8 * 2
                 + 2 * 7 * 8 * 2 + 7 * 8 * 2 + 10 * 8 * 2)


def test_chain_step_waits_for_each_input_before_its_first_reader(monkeypatch):
    """The end-to-end arm copies a step's inputs one by one; the step makes each
    operator wait only for the inputs it is the first to read, in reading order,
    and every per-step input is waited for exactly once."""
    import numpy as np
    import torch
    monkeypatch.setattr(bench, "HIDDEN", 8)
    monkeypatch.setattr(bench, "INTER", 12)
    monkeypatch.setattr(bench, "VOCAB", 10)
    S = 4
    inputs = {k: np.zeros(sh, np.float32) for k, sh in
              {"x": (S, 8), "w": (8,), "dy_r": (S, 8), "q": (1, S, 2, 4), "k": (1, S, 2, 4), "dq": (1, S, 2, 4),
               "dk": (1, S, 2, 4), "gate": (S, 12), "up": (S, 12), "dy_s": (S, 12), "X": (S, 8),
               "W": (10, 8)}.items()}
    inputs["labels"] = np.array([1, -100, 3, 4], np.int64)
    log = []
    ch = bench.Chain(_RecordingLib(log), inputs, torch.device("cpu"))
    ch.step(ready=lambda k: log.append(("ready", k, None)))
    seq = [e[1] if e[0] == "ready" else e[0] for e in log]
    assert seq == ["x", "liger_rmsnorm_fwd", "q", "k", "liger_rope_fwd", "gate", "up", "liger_swiglu_fwd",
                   "X", "labels", "liger_linear_ce_fwd_bwd", "dy_s", "liger_swiglu_bwd", "dq", "dk",
                   "liger_rope_bwd", "dy_r", "liger_rmsnorm_bwd"]
    waited = sorted(e[1] for e in log if e[0] == "ready")
    assert waited == sorted(k for k in inputs if k not in bench.PARAMETERS)
