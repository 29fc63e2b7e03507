"""The linear cross-entropies without their host wait (liger_linear_ce_fwd_bwd_async,
liger_linear_ce_two_pass_fwd_bwd_async), through the C-ABI: bit-identical to
the waiting forms when no label is ignored (tensor-core and fp32 SIMT paths,
both reductions); with ignored labels the waiting bf16 forms (token-chunked and
two-pass) run the other tokens only, so lse and dX stay bit-identical (each row is computed from
the same operands in the same order) while dW and the loss are sums over a
different grouping of the tokens, equal within rounding; a bad label is
treated as ignored and makes the loss NaN,
the gradients equal those of the same batch with that label ignored; an
all-ignored batch gives loss 0 and zero gradients; and the call can be
captured in a CUDA graph whose replay reproduces the eager results."""
import math

import numpy as np
import pytest

import datagen
from gpu_util import bits, dev

pytestmark = pytest.mark.gpu


def _call(L, X, W, lab, two_pass=False, wait=True, reduction="mean", grad_scale=1.0, chunk=0):
    import torch
    T, H = X.shape
    V = W.shape[0]
    code = L.LIGER_F32 if X.dtype == torch.float32 else L.LIGER_BF16
    n = (L.liger_linear_ce_two_pass_workspace(T, H, V, chunk) if two_pass
         else L.liger_linear_ce_workspace(T, H, V, chunk, code))
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
    loss = torch.full((1,), 7.0, dtype=torch.float32, device="cuda")
    dX, dW = torch.empty_like(X), torch.empty_like(W)
    if two_pass:
        L.liger_linear_ce_two_pass_fwd_bwd(X, W, lab, loss, dX, dW, ws, -100, reduction, grad_scale, chunk, wait=wait)
    else:
        L.liger_linear_ce_fwd_bwd(X, W, lab, loss, dX, dW, ws, -100, reduction, grad_scale, chunk, wait=wait)
    torch.cuda.synchronize()
    return loss, dX, dW, ws[: 4 * T].view(torch.float32).clone()


def _inputs(seed, T, H, V, dtype="bf16", frac=0.1):
    X = dev(datagen.normal(seed, "aX", (T, H), dtype))
    W = dev(datagen.normal(seed, "aW", (V, H), dtype, 0.0, 0.05))
    lab = dev(datagen.labels(seed, "al", T, V, frac))
    return X, W, lab


def _same(a, b):
    for x, y in zip(a, b):
        assert np.array_equal(bits(x), bits(y))


@pytest.mark.parametrize("T,H,V,dtype,two_pass,reduction,chunk", [
    (300, 320, 2037, "bf16", False, "mean", 128),
    (257, 136, 777, "bf16", False, "sum", 0),
    (9000, 64, 300, "bf16", False, "mean", 16384),   # several label-sort segments in one chunk
    (130, 64, 300, "f32", False, "mean", 0),          # fp32 SIMT path
    (300, 320, 2037, "bf16", True, "mean", 512),
    (129, 64, 256, "bf16", True, "sum", 0),
    (256, 64, 66536, "bf16", False, "mean", 0),       # dX over two vocabulary slabs
])
def test_async_matches_waiting_form(cuda_lib, T, H, V, dtype, two_pass, reduction, chunk):
    import oracle
    from gpu_util import host
    # no label ignored: bit-identical
    X, W, lab = _inputs(71, T, H, V, dtype, frac=0.0)
    a = _call(cuda_lib, X, W, lab, two_pass, True, reduction, 0.5, chunk)
    b = _call(cuda_lib, X, W, lab, two_pass, False, reduction, 0.5, chunk)
    _same(a, b)
    # 10 % ignored
    X, W, lab = _inputs(71, T, H, V, dtype)
    a = _call(cuda_lib, X, W, lab, two_pass, True, reduction, 0.5, chunk)
    b = _call(cuda_lib, X, W, lab, two_pass, False, reduction, 0.5, chunk)
    compacted = dtype == "bf16"
    if not compacted:
        _same(a, b)
        return
    _same((a[1], a[3]), (b[1], b[3]))                                   # dX, lse
    assert abs(float(a[0].item()) - float(b[0].item())) <= 1e-6 * abs(float(b[0].item()))
    assert oracle.rel_err(host(a[2]), host(b[2])) <= 1e-2               # dW: rounding of the sums only


@pytest.mark.parametrize("two_pass", [False, True])
def test_async_bad_labels_are_ignored_and_the_loss_is_nan(cuda_lib, two_pass):
    T, H, V = 300, 128, 1000
    X, W, lab = _inputs(72, T, H, V)
    bad = lab.clone()
    bad[3], bad[150], bad[299] = V, -5, 1 << 40
    fixed = bad.clone()
    fixed[3] = fixed[150] = fixed[299] = -100
    got = _call(cuda_lib, X, W, bad, two_pass, wait=False)
    want = _call(cuda_lib, X, W, fixed, two_pass, wait=True)
    assert math.isnan(got[0].item())
    # the waiting form runs the non-ignored tokens only: dW summed over another grouping
    import oracle
    from gpu_util import host
    _same((got[1], got[3]), (want[1], want[3]))
    assert oracle.rel_err(host(got[2]), host(want[2])) <= 1e-2
    with pytest.raises(cuda_lib.LigerError) as e:   # the waiting form refuses the batch
        _call(cuda_lib, X, W, bad, two_pass, wait=True)
    assert e.value.status == -5


@pytest.mark.parametrize("two_pass", [False, True])
def test_async_all_ignored(cuda_lib, two_pass):
    T, H, V = 256, 128, 512
    X, W, _ = _inputs(73, T, H, V)
    import torch
    lab = torch.full((T,), -100, dtype=torch.int64, device="cuda")
    loss, dX, dW, lse = _call(cuda_lib, X, W, lab, two_pass, wait=False)
    assert loss.item() == 0.0
    # dX and lse rows of ignored tokens are written +0; dW is the GEMM over an all-zero D
    assert np.all(bits(dX) == 0) and np.all(bits(lse) == 0) and bool((dW.float() == 0).all())


def test_async_capture_in_a_cuda_graph(cuda_lib):
    import torch
    T, H, V = 1000, 256, 5000
    X, W, lab = _inputs(74, T, H, V)
    ref = _call(cuda_lib, X, W, lab, wait=False)   # the same form, eager
    ws = torch.empty(cuda_lib.liger_linear_ce_workspace(T, H, V, 0, cuda_lib.LIGER_BF16), dtype=torch.uint8,
                     device="cuda")
    ws2 = torch.empty(cuda_lib.liger_linear_ce_two_pass_workspace(T, H, V, 0), dtype=torch.uint8, device="cuda")
    loss, loss2 = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    dX, dW, dX2, dW2 = torch.empty_like(X), torch.empty_like(W), torch.empty_like(X), torch.empty_like(W)

    def step():
        cuda_lib.liger_linear_ce_fwd_bwd(X, W, lab, loss, dX, dW, ws, wait=False)
        cuda_lib.liger_linear_ce_two_pass_fwd_bwd(X, W, lab, loss2, dX2, dW2, ws2, wait=False)

    step()   # first calls on the device, outside the capture
    ref2 = (loss2.clone(), dX2.clone(), dW2.clone())
    torch.cuda.synchronize()
    for t in (loss, dX, dW, loss2, dX2, dW2):
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    _same((loss, dX, dW), ref[:3])
    _same((loss2, dX2, dW2), ref2)
