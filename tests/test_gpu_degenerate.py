"""Degenerate sizes on the tensor-core paths, against the fp64 oracle: a single
token (one CTA pair whose second CTA holds only out-of-range rows), widths that
fill less than one 256-column tile, and the smallest hidden size the GEMMs take."""
import numpy as np
import pytest

import datagen
import oracle
from gpu_util import LOSS_TOL_BF16, TOL, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,H,V", [(1, 64, 256), (1, 128, 300), (2, 64, 257)])
def test_linear_ce_single_token(cuda_lib, T, H, V):
    import torch
    X = datagen.normal(71, "dX", (T, H), "bf16")
    W = datagen.normal(71, "dW", (V, H), "bf16", 0.0, 0.05)
    lab = np.arange(T, dtype=np.int64) % V
    o = oracle.linear_ce(X, W, lab)
    for two_pass in (False, True):
        n = (cuda_lib.liger_linear_ce_two_pass_workspace(T, H, V) if two_pass
             else cuda_lib.liger_linear_ce_workspace(T, H, V, 0, cuda_lib.LIGER_BF16))
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        loss = torch.empty(1, dtype=torch.float32, device="cuda")
        tX, tW = dev(X), dev(W)
        dX, dW = torch.empty_like(tX), torch.empty_like(tW)
        fn = cuda_lib.liger_linear_ce_two_pass_fwd_bwd if two_pass else cuda_lib.liger_linear_ce_fwd_bwd
        fn(tX, tW, dev(lab), loss, dX, dW, ws)
        torch.cuda.synchronize()
        assert abs(float(loss.item()) - o["loss"]) <= LOSS_TOL_BF16 * abs(o["loss"])
        assert oracle.rel_err(host(dX), o["dX"]) <= TOL["bf16"]
        assert oracle.rel_err(host(dW), o["dW"]) <= TOL["bf16"]


@pytest.mark.parametrize("T,H,I", [(1, 64, 8), (1, 64, 136), (3, 128, 264)])
def test_fused_linear_swiglu_tiny(cuda_lib, T, H, I):
    import torch
    X = datagen.normal(72, "tX", (T, H), "bf16")
    Wg = datagen.normal(72, "tg", (I, H), "bf16", 0.0, 0.05)
    Wu = datagen.normal(72, "tu", (I, H), "bf16", 0.0, 0.05)
    dH = datagen.normal(72, "td", (T, I), "bf16")
    tX, tg, tu = dev(X), dev(Wg), dev(Wu)
    h = torch.empty(T, I, dtype=torch.bfloat16, device="cuda")
    cuda_lib.liger_fused_linear_swiglu_fwd(tX, tg, tu, h)
    ws = torch.empty(cuda_lib.liger_fused_linear_swiglu_workspace(T, I), dtype=torch.uint8, device="cuda")
    dX, dWg, dWu = torch.empty_like(tX), torch.empty_like(tg), torch.empty_like(tu)
    cuda_lib.liger_fused_linear_swiglu_bwd(tX, tg, tu, dev(dH), dX, dWg, dWu, ws)
    torch.cuda.synchronize()
    assert oracle.rel_err(host(h), oracle.linear_swiglu_fwd(X, Wg, Wu)) <= TOL["bf16"]
    odX, odWg, odWu = oracle.linear_swiglu_bwd(X, Wg, Wu, dH)
    assert oracle.rel_err(host(dX), odX) <= TOL["bf16"]
    assert oracle.rel_err(host(dWg), odWg) <= TOL["bf16"]
    assert oracle.rel_err(host(dWu), odWu) <= TOL["bf16"]


def test_rmsnorm_qkv_rope_single_token(cuda_lib):
    import torch
    B, S, H, Hq, Hk, D = 1, 1, 64, 1, 1, 64
    x = datagen.normal(73, "sx", (B * S, H), "bf16")
    w = datagen.normal(73, "sw", (H,), "bf16", 1.0, 0.1)
    Wq, Wk, Wv = (datagen.normal(73, n, (D, H), "bf16", 0.0, 0.05) for n in ("sq", "sk", "sv"))
    pos = np.array([[12345]], np.int32)
    q = torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device="cuda")
    k, v = torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(cuda_lib.liger_rmsnorm_qkv_rope_workspace(1, H, Hq, Hk, D), dtype=torch.uint8, device="cuda")
    cuda_lib.liger_rmsnorm_qkv_rope_fwd(dev(x), dev(w), dev(Wq), dev(Wk), dev(Wv), q, k, v, ws, B, S, Hq, Hk, D,
                                        pos=dev(pos))
    torch.cuda.synchronize()
    oq, ok_, ov, _ = oracle.rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, 1e-6, 1e4, pos=pos)
    assert oracle.rel_err(host(q), oq) <= TOL["bf16"]
    assert oracle.rel_err(host(k), ok_) <= TOL["bf16"]
    assert oracle.rel_err(host(v), ov) <= TOL["bf16"]


@pytest.mark.parametrize("T,H,V,valid", [(1000, 128, 700, (517,)), (300, 64, 300, (0, 299)),
                                         (257, 64, 513, "all but 128")])
def test_linear_ce_compaction_extremes(cuda_lib, T, H, V, valid):
    """The waiting bf16 entry points run only the tokens whose label is not
    ignored: one valid token among a thousand (the run is a single row), the first
    and last tokens only, and every token but one; against the oracle, with the
    ignored rows of dX and lse exactly +0."""
    import torch
    X = datagen.normal(74, "cX", (T, H), "bf16")
    W = datagen.normal(74, "cW", (V, H), "bf16", 0.0, 0.05)
    lab = datagen.labels(74, "cl", T, V, 0.0)
    keep = np.zeros(T, bool)
    if valid == "all but 128":
        keep[:] = True
        keep[128] = False
    else:
        keep[list(valid)] = True
    lab[~keep] = -100
    o = oracle.linear_ce(X, W, lab)
    for two_pass in (False, True):
        n = (cuda_lib.liger_linear_ce_two_pass_workspace(T, H, V) if two_pass
             else cuda_lib.liger_linear_ce_workspace(T, H, V, 0, cuda_lib.LIGER_BF16))
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        loss = torch.empty(1, dtype=torch.float32, device="cuda")
        tX, tW = dev(X), dev(W)
        dX, dW = torch.full_like(tX, 7.0), torch.empty_like(tW)
        fn = cuda_lib.liger_linear_ce_two_pass_fwd_bwd if two_pass else cuda_lib.liger_linear_ce_fwd_bwd
        fn(tX, tW, dev(lab), loss, dX, dW, ws)
        torch.cuda.synchronize()
        assert abs(float(loss.item()) - o["loss"]) <= LOSS_TOL_BF16 * abs(o["loss"])
        hdX = host(dX)
        assert oracle.rel_err(hdX, o["dX"]) <= TOL["bf16"]
        assert np.all(hdX[~keep] == 0) and not np.any(np.signbit(hdX[~keep]))
        assert oracle.rel_err(host(dW), o["dW"]) <= TOL["bf16"]
        lse = host(ws[: 4 * T].view(torch.float32))
        assert np.all(lse[~keep] == 0)
        assert oracle.rel_err(lse[keep], o["lse"][keep]) <= 1e-3
