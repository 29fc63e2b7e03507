"""Calls from several host threads at once, in a fresh process: the library's
lazily initialised per-device state (GEMM attributes and occupancy, the tensor-map
encoder, error words) is set up by whichever thread comes first while the others
race it.  Four threads released together by a barrier each run the linear
cross-entropy, FusedLinearSwiGLU and the fused QKV projection on their own
stream and buffers; the kernels are deterministic, so every thread's results
must be bit-identical."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import transformer_rmsnorm_fwd_gb300 as L

N = 4
gate = threading.Barrier(N)
out = [None] * N
errs = []

def work(i):
    try:
        torch.cuda.set_device(0)
        g = torch.Generator(device="cuda").manual_seed(7)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            T, H, V = 512, 256, 4096
            X = torch.randn(T, H, device="cuda", generator=g).bfloat16()
            W = (torch.randn(V, H, device="cuda", generator=g) * 0.05).bfloat16()
            lab = torch.randint(0, V, (T,), device="cuda", generator=g)
            ws = torch.empty(L.liger_linear_ce_workspace(T, H, V), dtype=torch.uint8, device="cuda")
            loss = torch.empty(1, device="cuda")
            dX, dW = torch.empty_like(X), torch.empty_like(W)
            I = 512
            Wg = (torch.randn(I, H, device="cuda", generator=g) * 0.05).bfloat16()
            Wu = (torch.randn(I, H, device="cuda", generator=g) * 0.05).bfloat16()
            h = torch.empty(T, I, device="cuda", dtype=torch.bfloat16)
            Hq, D = 2, 64
            wn = torch.ones(H, device="cuda", dtype=torch.bfloat16)
            Wq = (torch.randn(Hq * D, H, device="cuda", generator=g) * 0.05).bfloat16()
            q = torch.empty(1, T, Hq, D, device="cuda", dtype=torch.bfloat16)
            k, v = torch.empty_like(q), torch.empty_like(q)
            wq = torch.empty(L.liger_rmsnorm_qkv_rope_workspace(T, H, Hq, Hq, D), dtype=torch.uint8, device="cuda")
            s.synchronize()
            gate.wait()
            L.liger_linear_ce_fwd_bwd(X, W, lab, loss, dX, dW, ws)
            L.liger_fused_linear_swiglu_fwd(X, Wg, Wu, h)
            L.liger_rmsnorm_qkv_rope_fwd(X, wn, Wq, Wq, Wq, q, k, v, wq, 1, T, Hq, Hq, D)
            s.synchronize()
        out[i] = [t.view(torch.int16).cpu() if t.dtype == torch.bfloat16 else t.cpu() for t in (loss, dX, dW, h, q, k, v)]
    except Exception as e:
        errs.append(repr(e))

ts = [threading.Thread(target=work, args=(i,)) for i in range(N)]
for t in ts: t.start()
for t in ts: t.join()
assert not errs, errs
for i in range(1, N):
    for a, b in zip(out[0], out[i]):
        assert torch.equal(a, b), i
print("threads ok")
"""


def test_concurrent_first_calls_from_host_threads(cuda_lib):
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
