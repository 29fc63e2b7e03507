"""GPU parity of FusedLinearSwiGLU (forward and backward) against the fp64
oracle, through the C-ABI: ragged shapes whose T, H and I are not multiples
of the 256 x 256 x 64 tensor-core (CTA-pair) tiles, and the pages' configuration (hidden
4096, intermediate 11008, 4 x 2048 tokens) on sampled rows."""
import numpy as np
import pytest

import datagen
import oracle
from gpu_util import dev, host

pytestmark = pytest.mark.gpu


def _run(L, X, Wg, Wu, dH):
    import torch
    tX, tg, tu = dev(X), dev(Wg), dev(Wu)
    T, H = X.shape
    I = Wg.shape[0]
    out = torch.empty(T, I, dtype=torch.bfloat16, device="cuda")
    L.liger_fused_linear_swiglu_fwd(tX, tg, tu, out)
    ws = torch.empty(L.liger_fused_linear_swiglu_workspace(T, I), dtype=torch.uint8, device="cuda")
    dX, dWg, dWu = torch.empty_like(tX), torch.empty_like(tg), torch.empty_like(tu)
    L.liger_fused_linear_swiglu_bwd(tX, tg, tu, dev(dH), dX, dWg, dWu, ws)
    torch.cuda.synchronize()
    return out, dX, dWg, dWu


@pytest.mark.parametrize("T,H,I", [(300, 320, 688), (129, 64, 128), (64, 256, 8), (512, 512, 1000)])
def test_fused_linear_swiglu_ragged(cuda_lib, T, H, I):
    X = datagen.normal(51, "sx", (T, H), "bf16")
    Wg = datagen.normal(51, "sg", (I, H), "bf16", 0.0, 0.05)
    Wu = datagen.normal(51, "su", (I, H), "bf16", 0.0, 0.05)
    dH = datagen.normal(51, "sd", (T, I), "bf16")
    out, dX, dWg, dWu = _run(cuda_lib, X, Wg, Wu, dH)
    assert oracle.rel_err(host(out), oracle.linear_swiglu_fwd(X, Wg, Wu)) <= 2e-2
    odX, odWg, odWu = oracle.linear_swiglu_bwd(X, Wg, Wu, dH)
    assert oracle.rel_err(host(dX), odX) <= 2e-2
    assert oracle.rel_err(host(dWg), odWg) <= 2e-2
    assert oracle.rel_err(host(dWu), odWu) <= 2e-2


def test_fused_linear_swiglu_llama_mlp_sampled(cuda_lib):
    """T = 4 x 2048, hidden 4096, intermediate 11008 (the pages' SwiGLU configuration):
    forward rows and dX rows sampled against the oracle."""
    T, H, I = 8192, 4096, 11008
    X = datagen.normal(52, "mx", (T, H), "bf16")
    Wg = datagen.normal(52, "mg", (I, H), "bf16", 0.0, 0.02)
    Wu = datagen.normal(52, "mu", (I, H), "bf16", 0.0, 0.02)
    dH = datagen.normal(52, "md", (T, I), "bf16")
    out, dX, dWg, dWu = _run(cuda_lib, X, Wg, Wu, dH)
    rows = np.array([0, 1, 4097, 8191])
    ho, hdx = host(out), host(dX)
    assert oracle.rel_err(ho[rows], oracle.linear_swiglu_fwd(X[rows], Wg, Wu)) <= 2e-2
    odX, _, _ = oracle.linear_swiglu_bwd(X[rows], Wg, Wu, dH[rows])
    assert oracle.rel_err(hdx[rows], odX) <= 2e-2
    # a row of dW_g / dW_u depends only on its own intermediate column, so the
    # oracle restricted to sampled columns gives those rows exactly
    cols = np.array([0, 257, 5504, 11007])
    _, odWg, odWu = oracle.linear_swiglu_bwd(X, Wg[cols], Wu[cols], dH[:, cols])
    assert oracle.rel_err(host(dWg)[cols], odWg) <= 2e-2
    assert oracle.rel_err(host(dWu)[cols], odWu) <= 2e-2


def test_fused_linear_swiglu_empty_tokens(cuda_lib):
    import torch
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.ones(16, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(0, 16, dtype=torch.bfloat16, device="cuda")
    cuda_lib.liger_fused_linear_swiglu_fwd(X, W, W, out)
    dWg, dWu = torch.ones_like(W), torch.ones_like(W)
    ws = torch.empty(max(1, cuda_lib.liger_fused_linear_swiglu_workspace(0, 16)), dtype=torch.uint8, device="cuda")
    cuda_lib.liger_fused_linear_swiglu_bwd(X, W, W, out, torch.empty_like(X), dWg, dWu, ws)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(dWg)) == 0 and int(torch.count_nonzero(dWu)) == 0


def test_fused_linear_swiglu_errors(cuda_lib):
    import torch
    X = torch.zeros(8, 64, dtype=torch.float32, device="cuda")
    W = torch.zeros(16, 64, dtype=torch.float32, device="cuda")
    out = torch.empty(8, 16, dtype=torch.float32, device="cuda")
    with pytest.raises(cuda_lib.LigerError) as e:
        cuda_lib.liger_fused_linear_swiglu_fwd(X, W, W, out)
    assert e.value.status == -3
    Xb = torch.zeros(8, 60, dtype=torch.bfloat16, device="cuda")
    Wb = torch.zeros(16, 60, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.LigerError) as e:
        cuda_lib.liger_fused_linear_swiglu_fwd(Xb, Wb, Wb, out.bfloat16())
    assert e.value.status == -2


def _run_saved(L, X, Wg, Wu, dH):
    import torch
    tX, tg, tu = dev(X), dev(Wg), dev(Wu)
    T, H = X.shape
    I = Wg.shape[0]
    out = torch.empty(T, I, dtype=torch.bfloat16, device="cuda")
    g, u = torch.empty_like(out), torch.empty_like(out)
    L.liger_fused_linear_swiglu_fwd_save(tX, tg, tu, out, g, u)
    ws = torch.empty(L.liger_fused_linear_swiglu_workspace(T, I), dtype=torch.uint8, device="cuda")
    dX, dWg, dWu = torch.empty_like(tX), torch.empty_like(tg), torch.empty_like(tu)
    L.liger_fused_linear_swiglu_bwd_saved(tX, tg, tu, dev(dH), g, u, dX, dWg, dWu, ws)
    torch.cuda.synchronize()
    return out, g, u, dX, dWg, dWu


@pytest.mark.parametrize("T,H,I", [(300, 320, 688), (129, 64, 128), (64, 256, 8)])
def test_fused_linear_swiglu_saved_ragged(cuda_lib, T, H, I):
    """The saving forward writes h and the exact-up-to-rounding g = X Wg^T, u = X Wu^T;
    the backward from them matches the oracle."""
    X = datagen.normal(53, "vx", (T, H), "bf16")
    Wg = datagen.normal(53, "vg", (I, H), "bf16", 0.0, 0.05)
    Wu = datagen.normal(53, "vu", (I, H), "bf16", 0.0, 0.05)
    dH = datagen.normal(53, "vd", (T, I), "bf16")
    out, g, u, dX, dWg, dWu = _run_saved(cuda_lib, X, Wg, Wu, dH)
    xf, gf, uf = (datagen.to_f64(a, "bf16") for a in (X, Wg, Wu))
    assert oracle.rel_err(host(g), xf @ gf.T) <= 2e-2 and oracle.rel_err(host(u), xf @ uf.T) <= 2e-2
    assert oracle.rel_err(host(out), oracle.linear_swiglu_fwd(X, Wg, Wu)) <= 2e-2
    odX, odWg, odWu = oracle.linear_swiglu_bwd(X, Wg, Wu, dH)
    assert oracle.rel_err(host(dX), odX) <= 2e-2
    assert oracle.rel_err(host(dWg), odWg) <= 2e-2
    assert oracle.rel_err(host(dWu), odWu) <= 2e-2


def test_fused_linear_swiglu_saved_llama_mlp_sampled(cuda_lib):
    """T = 4 x 2048, hidden 4096, intermediate 11008: sampled rows of h and dX,
    sampled intermediate columns of dW_g and dW_u against the oracle."""
    T, H, I = 8192, 4096, 11008
    X = datagen.normal(52, "mx", (T, H), "bf16")
    Wg = datagen.normal(52, "mg", (I, H), "bf16", 0.0, 0.02)
    Wu = datagen.normal(52, "mu", (I, H), "bf16", 0.0, 0.02)
    dH = datagen.normal(52, "md", (T, I), "bf16")
    out, g, u, dX, dWg, dWu = _run_saved(cuda_lib, X, Wg, Wu, dH)
    rows = np.array([0, 1, 4097, 8191])
    assert oracle.rel_err(host(out)[rows], oracle.linear_swiglu_fwd(X[rows], Wg, Wu)) <= 2e-2
    odX, _, _ = oracle.linear_swiglu_bwd(X[rows], Wg, Wu, dH[rows])
    assert oracle.rel_err(host(dX)[rows], odX) <= 2e-2
    cols = np.array([0, 257, 5504, 11007])
    _, odWg, odWu = oracle.linear_swiglu_bwd(X, Wg[cols], Wu[cols], dH[:, cols])
    assert oracle.rel_err(host(dWg)[cols], odWg) <= 2e-2
    assert oracle.rel_err(host(dWu)[cols], odWu) <= 2e-2


def test_fused_linear_swiglu_l2_sized_launches(cuda_lib):
    """The forward and the backward's recompute GEMM run over at most 32 MiB of
    X rows per launch (8192 rows at hidden 2048): T = 9000 takes a full and a
    ragged launch; the dW GEMMs take the grouped tile order (X above 32 MiB).
    Forward, backward and the saving pair against the oracle."""
    T, H, I = 9000, 2048, 64
    X = datagen.normal(54, "lx", (T, H), "bf16")
    Wg = datagen.normal(54, "lg", (I, H), "bf16", 0.0, 0.02)
    Wu = datagen.normal(54, "lu", (I, H), "bf16", 0.0, 0.02)
    dH = datagen.normal(54, "ld", (T, I), "bf16")
    out, dX, dWg, dWu = _run(cuda_lib, X, Wg, Wu, dH)
    assert oracle.rel_err(host(out), oracle.linear_swiglu_fwd(X, Wg, Wu)) <= 2e-2
    odX, odWg, odWu = oracle.linear_swiglu_bwd(X, Wg, Wu, dH)
    assert oracle.rel_err(host(dX), odX) <= 2e-2
    assert oracle.rel_err(host(dWg), odWg) <= 2e-2
    assert oracle.rel_err(host(dWu), odWu) <= 2e-2
    # the saving pair: h as above; its backward is the exact backward from the g, u it
    # stored (bf16: one rounding more than the recompute path, which over 18 M elements
    # reaches 2.5 % of rms against the oracle's unrounded g, u)
    out2, g, u, dX2, dWg2, dWu2 = _run_saved(cuda_lib, X, Wg, Wu, dH)
    assert np.array_equal(host(out2), host(out))
    dGr, dUr = oracle.swiglu_bwd(datagen.to_f64(dH, "bf16"), host(g), host(u))
    xf, gf, uf = (datagen.to_f64(a, "bf16") for a in (X, Wg, Wu))
    assert oracle.rel_err(host(dX2), dGr @ gf + dUr @ uf) <= 2e-2
    assert oracle.rel_err(host(dWg2), dGr.T @ xf) <= 2e-2
    assert oracle.rel_err(host(dWu2), dUr.T @ xf) <= 2e-2
