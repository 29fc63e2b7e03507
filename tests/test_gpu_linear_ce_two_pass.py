"""GPU parity of the two-pass, vocabulary-chunked fused linear cross-entropy
against the fp64 oracle, through the C-ABI: ragged shapes over several
vocabulary chunks (a short last chunk, chunk widths that are not multiples of
the 256-wide tile), more tokens than one label-sort segment (8192), sum
reduction with a gradient scale, the all-ignored batch, error codes, the
per-row forward shared bit for bit with the token-chunked path, and the
Qwen-7B head (seq 32768 x hidden 4096 x vocab 151936) on sampled rows."""
import math

import numpy as np
import pytest

import datagen
import oracle
from conftest import golden
from gpu_util import LOSS_TOL_BF16, TOL, bits, dev, host

pytestmark = pytest.mark.gpu


def _run(L, X, W, lab, vchunk=0, reduction="mean", grad_scale=1.0, two_pass=True):
    import torch
    tX, tW, tl = dev(X), dev(W), dev(lab)
    T, H = X.shape
    V = W.shape[0]
    n = (L.liger_linear_ce_two_pass_workspace(T, H, V, vchunk) if two_pass
         else L.liger_linear_ce_workspace(T, H, V, 0, L.LIGER_BF16))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    dX, dW = torch.empty_like(tX), torch.empty_like(tW)
    if two_pass:
        L.liger_linear_ce_two_pass_fwd_bwd(tX, tW, tl, loss, dX, dW, ws, -100, reduction, grad_scale, vchunk)
    else:
        L.liger_linear_ce_fwd_bwd(tX, tW, tl, loss, dX, dW, ws, -100, reduction, grad_scale)
    torch.cuda.synchronize()
    off = (4 * T + 255) // 256 * 256          # loss_row starts at the next 256-byte boundary
    lse = ws[: 4 * T].view(torch.float32).cpu().numpy().astype(np.float64)
    lrow = ws[off: off + 4 * T].view(torch.float32).cpu().numpy().astype(np.float64)
    return float(loss.item()), dX, dW, lse, lrow


def _check(X, W, lab, res, reduction="mean", grad_scale=1.0):
    loss, dX, dW, lse, _ = res
    o = oracle.linear_ce(X, W, lab, reduction=reduction, grad_scale=grad_scale)
    assert abs(loss - o["loss"]) <= LOSS_TOL_BF16 * abs(o["loss"]), (loss, o["loss"])
    assert oracle.rel_err(host(dX), o["dX"]) <= TOL["bf16"]
    assert oracle.rel_err(host(dW), o["dW"]) <= TOL["bf16"]
    assert oracle.rel_err(lse, o["lse"]) <= 1e-5
    ign = lab == -100
    assert np.all(bits(dX)[ign] == 0) and np.all(lse[ign] == 0)


@pytest.mark.parametrize("T,H,V,vchunk", [
    (300, 320, 2037, 512),    # 4 vocabulary chunks, the last 501 rows wide
    (129, 64, 256, 0),        # one chunk: dX written without the fp32 accumulator
    (1000, 512, 5000, 1000),  # chunk width not a multiple of the 256-wide tile
    (257, 136, 777, 264),
    (9000, 64, 300, 128),     # two label-sort segments, two pass-1 token chunks
])
def test_linear_ce_two_pass_ragged(cuda_lib, T, H, V, vchunk):
    X = datagen.normal(31, "tX", (T, H), "bf16")
    W = datagen.normal(31, "tW", (V, H), "bf16", 0.0, 0.05)
    lab = datagen.labels(31, "tl", T, V, 0.1)
    _check(X, W, lab, _run(cuda_lib, X, W, lab, vchunk))


def test_linear_ce_two_pass_repeated_labels(cuda_lib):
    """Few distinct labels, so many tokens share each dW row's one-hot correction
    (spread over both label-sort segments)."""
    T, H, V = 8300, 64, 256
    X = datagen.normal(32, "rX", (T, H), "bf16")
    W = datagen.normal(32, "rW", (V, H), "bf16", 0.0, 0.05)
    lab = datagen.labels(32, "rl", T, 3, 0.05)     # labels in {0, 1, 2}
    _check(X, W, lab, _run(cuda_lib, X, W, lab, 256))


def test_linear_ce_two_pass_sum_and_scale(cuda_lib):
    T, H, V = 130, 128, 512
    X = datagen.normal(33, "sX", (T, H), "bf16")
    W = datagen.normal(33, "sW", (V, H), "bf16", 0.0, 0.05)
    lab = datagen.labels(33, "sl", T, V, 0.1)
    _check(X, W, lab, _run(cuda_lib, X, W, lab, 256, reduction="sum", grad_scale=0.5), reduction="sum",
           grad_scale=0.5)


def test_linear_ce_two_pass_forward_matches_token_chunked(cuda_lib):
    """Pass 1 runs the same logits GEMM and merge as the token-chunked path:
    lse, the loss terms and the loss are bit-identical."""
    T, H, V = 700, 256, 3000
    X = datagen.normal(34, "mX", (T, H), "bf16")
    W = datagen.normal(34, "mW", (V, H), "bf16", 0.0, 0.05)
    lab = datagen.labels(34, "ml", T, V, 0.1)
    a = _run(cuda_lib, X, W, lab, 512)
    b = _run(cuda_lib, X, W, lab, two_pass=False)
    assert np.array_equal(a[3], b[3]) and np.array_equal(a[4], b[4]) and a[0] == b[0]


def test_linear_ce_two_pass_all_ignored_and_errors(cuda_lib):
    import torch
    T, H, V = 256, 128, 512
    X = datagen.normal(35, "aX", (T, H), "bf16")
    W = datagen.normal(35, "aW", (V, H), "bf16", 0.0, 0.02)
    loss, dX, dW, lse, _ = _run(cuda_lib, X, W, np.full(T, -100, np.int64), 256)
    assert loss == 0.0 and np.all(bits(dX) == 0) and np.all(bits(dW) == 0) and np.all(lse == 0)
    tX, tW = dev(X), dev(W)
    lab = datagen.labels(35, "al", T, V, 0.0)
    lab[7] = V
    ws = torch.empty(cuda_lib.liger_linear_ce_two_pass_workspace(T, H, V, 0), dtype=torch.uint8, device="cuda")
    lossb = torch.full((1,), 7.0, device="cuda")
    with pytest.raises(cuda_lib.LigerError) as e:
        cuda_lib.liger_linear_ce_two_pass_fwd_bwd(tX, tW, dev(lab), lossb, None, None, ws)
    assert e.value.status == -5
    with pytest.raises(cuda_lib.LigerError) as e:
        cuda_lib.liger_linear_ce_two_pass_fwd_bwd(tX, tW, dev(lab), lossb, None, None, ws, vchunk=100)
    assert e.value.status == -2
    with pytest.raises(cuda_lib.LigerError) as e:
        cuda_lib.liger_linear_ce_two_pass_fwd_bwd(tX.float(), tW.float(), dev(lab), lossb, None, None, ws)
    assert e.value.status == -3
    torch.cuda.synchronize()
    assert lossb.item() == 7.0


def test_linear_ce_two_pass_qwen7b_seq32768_sampled(cuda_lib):
    """The Qwen-7B head of the benchmark's chain (seq 32768, hidden 4096, vocab
    151936, 10 % ignored, so the ignored tokens are dropped before both passes),
    auto vocabulary chunk: the mean loss and the lse of every token against the
    oracle's full forward (cached in tests/golden); 16 or more rows of dW (labels
    of tokens across the sequence, random rows, the first and last) against the
    oracle given that lse; the oracle on sampled rows (lse, loss term, dX row); the
    loss is the mean of the row terms and close to its Gaussian-logit value; dW
    rows sum to ~0 over the vocabulary; ignored rows exact zeros."""
    from datagen import workloads
    c = workloads.qwen_chain(32768)["linear_ce"]
    X, W, lab = c.make("X"), c.make("W"), c.make("labels")
    T, H = X.shape
    V = W.shape[0]
    loss, dX, dW, lse, lrow = _run(cuda_lib, X, W, lab)
    g = golden("linear_ce_qwen32768_lse.json")
    st = g["lse_row_stride"]
    olse = np.array(g["lse"])
    keep = lab[::st] != -100
    assert np.max(np.abs(lse[::st][keep] - olse[keep]) / np.abs(olse[keep])) <= 1e-5
    assert abs(loss - g["loss_mean"]) <= LOSS_TOL_BF16 * abs(g["loss_mean"])
    if st == 1:
        # rows of dW (each finished in one pass over all valid tokens of its vocabulary chunk)
        lab_rows = [int(lab[t]) for t in (3, 8200, 16390, 32760) if lab[t] >= 0]
        vrows = np.unique(np.concatenate([lab_rows, np.random.default_rng(7).choice(V, 14, replace=False),
                                          [0, V - 1]]))
        assert len(vrows) >= 16
        odW = oracle.linear_ce_dw_rows(X, W, lab, olse, vrows)
        import torch
        assert oracle.rel_err(host(dW[torch.as_tensor(vrows, device="cuda")]), odW) <= 2e-2
    n_valid = int((lab != -100).sum())
    assert abs(loss - lrow.sum() / n_valid) <= 1e-5 * abs(loss)
    rows = np.array([0, 8191, 8192, 32767])
    o = oracle.linear_ce_rows(X, W, lab, rows)
    hdX = host(dX)
    for i, r in enumerate(rows):
        if lab[r] == -100:
            assert lse[r] == 0 and np.all(bits(dX)[r] == 0)
            continue
        assert abs(lse[r] - o["lse"][i]) <= 1e-5 * abs(o["lse"][i])
        assert abs(lrow[r] - o["loss_term"][i]) <= 1e-3 * abs(o["loss_term"][i])
        assert oracle.rel_err(hdX[r], o["dX"][i]) <= 2e-2
    xf = datagen.to_f64(X, "bf16")
    valid = lab != -100
    expect = math.log(V) + float(np.mean(0.5 * 0.02 ** 2 * np.sum(xf[valid] ** 2, axis=1)))
    assert abs(loss - expect) < 0.06, (loss, expect)
    assert np.all(bits(dX)[~valid] == 0)
    dWd = dW.double()
    assert float(dWd.sum(0).abs().max()) <= 2e-2 * float(dWd.abs().sum(0).max())
