"""GPU parity of the fused RMSNorm + QKV projection + RoPE forward against the
fp64 oracle, through the C-ABI: ragged token counts that leave a partial
128-row tile, hidden sizes that are not multiples of the 64-wide k-block,
grouped k/v heads, every head_dim the kernel takes, biases, explicit
positions, caller cos/sin tables, reuse of the folded weights, and the
Qwen-7B layer shapes (hidden 4096, 32 heads of 128, QKV bias) at seq 32768
on sampled tokens."""
import numpy as np
import pytest

import datagen
import oracle
from gpu_util import TOL, bits, dev, host

pytestmark = pytest.mark.gpu


def _inputs(seed, B, S, H, Hq, Hk, D, bias=True):
    x = datagen.normal(seed, "qx", (B * S, H), "bf16")
    w = datagen.normal(seed, "qw", (H,), "bf16", 1.0, 0.1)
    Wq = datagen.normal(seed, "qWq", (Hq * D, H), "bf16", 0.0, 0.02)
    Wk = datagen.normal(seed, "qWk", (Hk * D, H), "bf16", 0.0, 0.02)
    Wv = datagen.normal(seed, "qWv", (Hk * D, H), "bf16", 0.0, 0.02)
    b = [datagen.normal(seed, n, (m,), "bf16", 0.0, 0.1) if bias else None
         for n, m in (("qbq", Hq * D), ("qbk", Hk * D), ("qbv", Hk * D))]
    return x, w, Wq, Wk, Wv, b


def _run(L, x, w, Wq, Wk, Wv, b, B, S, Hq, Hk, D, eps, theta, pos=None, cos_tab=None, sin_tab=None, ws=None,
         folded=False, dev_w=None):
    import torch
    T, H = x.shape
    q = torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(B, S, Hk, D, dtype=torch.bfloat16, device="cuda")
    v = torch.empty(B, S, Hk, D, dtype=torch.bfloat16, device="cuda")
    rstd = torch.empty(T, dtype=torch.float32, device="cuda")
    if ws is None:
        ws = torch.empty(L.liger_rmsnorm_qkv_rope_workspace(T, H, Hq, Hk, D), dtype=torch.uint8, device="cuda")
    tw = dev_w if dev_w is not None else [None if a is None else dev(a) for a in (w, Wq, Wk, Wv, *b)]
    L.liger_rmsnorm_qkv_rope_fwd(dev(x), tw[0], tw[1], tw[2], tw[3], q, k, v, ws, B, S, Hq, Hk, D,
                                 bq=tw[4], bk=tw[5], bv=tw[6], pos=None if pos is None else dev(pos),
                                 cos_tab=None if cos_tab is None else dev(cos_tab),
                                 sin_tab=None if sin_tab is None else dev(sin_tab), rstd=rstd, eps=eps, theta=theta,
                                 folded=folded)
    torch.cuda.synchronize()
    return q, k, v, rstd, ws


def _check(got, want):
    q, k, v, rstd = got
    oq, ok_, ov, orstd = want
    assert oracle.rel_err(host(q), oq) <= TOL["bf16"]
    assert oracle.rel_err(host(k), ok_) <= TOL["bf16"]
    assert oracle.rel_err(host(v), ov) <= TOL["bf16"]
    assert oracle.rel_err(host(rstd), orstd) <= TOL["f32"]


@pytest.mark.parametrize("B,S,H,Hq,Hk,D,bias", [
    (2, 75, 320, 4, 2, 64, True),       # T = 150: one full and one partial row tile; GQA, k and v share a tile
    (1, 300, 256, 2, 2, 128, False),    # no bias
    (1, 129, 520, 1, 1, 256, True),     # head_dim 256, hidden not a multiple of 64
    (3, 17, 64, 3, 1, 128, True),       # odd head counts: q and k share a tile, N = 640 ends in a half tile
    (1, 40, 64, 0, 2, 64, True),        # no q heads
    (1, 40, 64, 2, 0, 64, True),        # no k / v heads
])
def test_rmsnorm_qkv_rope_ragged(cuda_lib, B, S, H, Hq, Hk, D, bias):
    x, w, Wq, Wk, Wv, b = _inputs(61, B, S, H, Hq, Hk, D, bias)
    pos = datagen.positions(61, "qpos", (B, S), 65536)
    got = _run(cuda_lib, x, w, Wq, Wk, Wv, b, B, S, Hq, Hk, D, 1e-6, 1e4, pos=pos)[:4]
    want = oracle.rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, 1e-6, 1e4, *b, pos=pos)
    _check(got, want)


def test_rmsnorm_qkv_rope_default_positions_and_theta(cuda_lib):
    B, S, H, Hq, Hk, D = 2, 40, 128, 2, 1, 64
    x, w, Wq, Wk, Wv, b = _inputs(62, B, S, H, Hq, Hk, D)
    got = _run(cuda_lib, x, w, Wq, Wk, Wv, b, B, S, Hq, Hk, D, 1e-5, 5e5)[:4]
    _check(got, oracle.rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, 1e-5, 5e5, *b))


def test_rmsnorm_qkv_rope_caller_tables(cuda_lib):
    """cos/sin tables of a scaled schedule (positions / 4), indexed by position."""
    B, S, H, Hq, Hk, D, n_tab = 1, 96, 192, 2, 2, 128, 512
    x, w, Wq, Wk, Wv, b = _inputs(63, B, S, H, Hq, Hk, D)
    pos = datagen.positions(63, "tpos", (B, S), n_tab)
    p = np.arange(n_tab, dtype=np.float64)[:, None] / 4.0
    ang = p * 1e4 ** (-2.0 * np.arange(D // 2)[None, :] / D)
    ct, st = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    got = _run(cuda_lib, x, w, Wq, Wk, Wv, b, B, S, Hq, Hk, D, 1e-6, 1e4, pos=pos, cos_tab=ct, sin_tab=st)[:4]
    want = oracle.rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, 1e-6, 1e4, *b, pos=pos, cos_tab=ct, sin_tab=st)
    _check(got, want)


def test_rmsnorm_qkv_rope_folded_weights_reused(cuda_lib):
    """flags bit 0: the folded weights already in the workspace are used, the
    weight pointers are not read; results are bit-identical."""
    B, S, H, Hq, Hk, D = 1, 200, 256, 2, 1, 128
    x, w, Wq, Wk, Wv, b = _inputs(64, B, S, H, Hq, Hk, D)
    q1, k1, v1, r1, ws = _run(cuda_lib, x, w, Wq, Wk, Wv, b, B, S, Hq, Hk, D, 1e-6, 1e4)
    q2, k2, v2, r2, _ = _run(cuda_lib, x, w, Wq, Wk, Wv, b, B, S, Hq, Hk, D, 1e-6, 1e4, ws=ws, folded=True,
                             dev_w=[None] * 7)
    for a, c in ((q1, q2), (k1, k2), (v1, v2), (r1, r2)):
        assert np.array_equal(bits(a), bits(c))


def test_rmsnorm_qkv_rope_qwen7b_seq32768_sampled(cuda_lib):
    """Qwen-7B layer shapes (hidden 4096, 32 q and 32 k/v heads of 128, QKV bias)
    at batch 1, seq 32768, theta 1e4: sampled tokens against the oracle, and
    finite outputs everywhere."""
    import torch
    B, S, H, Hq, Hk, D = 1, 32768, 4096, 32, 32, 128
    x, w, Wq, Wk, Wv, b = _inputs(65, B, S, H, Hq, Hk, D)
    q, k, v, rstd, _ = _run(cuda_lib, x, w, Wq, Wk, Wv, b, B, S, Hq, Hk, D, 1e-6, 1e4)
    rows = np.array([0, 1, 127, 128, 16385, 32767])
    pos = rows.astype(np.int32).reshape(1, -1)
    want = oracle.rmsnorm_qkv_rope(x[rows], w, Wq, Wk, Wv, 1, len(rows), Hq, Hk, 1e-6, 1e4, *b, pos=pos)
    got = (q[0, rows], k[0, rows], v[0, rows], rstd[rows])
    q_, k_, v_, r_ = got
    assert oracle.rel_err(host(q_), want[0][0]) <= TOL["bf16"]
    assert oracle.rel_err(host(k_), want[1][0]) <= TOL["bf16"]
    assert oracle.rel_err(host(v_), want[2][0]) <= TOL["bf16"]
    assert oracle.rel_err(host(r_), want[3]) <= TOL["f32"]
    for t in (q, k, v):
        assert bool(torch.isfinite(t).all())


def test_rmsnorm_qkv_rope_empty_and_errors(cuda_lib):
    import torch
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(256, cuda_lib.liger_rmsnorm_qkv_rope_workspace(0, 64, 1, 1, 64)), dtype=torch.uint8,
                     device="cuda")
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    wn = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    e = torch.empty(1, 0, 1, 64, dtype=torch.bfloat16, device="cuda")
    cuda_lib.liger_rmsnorm_qkv_rope_fwd(x, wn, W, W, W, e, e, e, ws, 1, 0, 1, 1, 64)
    xf = torch.zeros(4, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(cuda_lib.LigerError) as err:
        cuda_lib.liger_rmsnorm_qkv_rope_fwd(xf, wn, W, W, W, e, e, e, ws, 1, 4, 1, 1, 64)
    assert err.value.status == -3


def test_rmsnorm_qkv_rope_caller_tables_without_positions_over_batches(cuda_lib):
    """Caller cos/sin tables and no positions, two sequences of 4500 tokens at
    hidden 2048: every token indexes the tables by its position in its own
    sequence (token % seq), across the batch boundary and beyond 8192 rows;
    sampled tokens against the oracle."""
    B, S, H, Hq, Hk, D, n_tab = 2, 4500, 2048, 1, 1, 64, 4500
    x, w, Wq, Wk, Wv, b = _inputs(66, B, S, H, Hq, Hk, D)
    p = np.arange(n_tab, dtype=np.float64)[:, None] / 2.0
    ang = p * 1e4 ** (-2.0 * np.arange(D // 2)[None, :] / D)
    ct, st = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    q, k, v, rstd, _ = _run(cuda_lib, x, w, Wq, Wk, Wv, b, B, S, Hq, Hk, D, 1e-6, 1e4, cos_tab=ct, sin_tab=st)
    rows = np.array([0, 4499, 4500, 8191, 8192, 8999])
    pos = (rows % S).astype(np.int32).reshape(1, -1)
    want = oracle.rmsnorm_qkv_rope(x[rows], w, Wq, Wk, Wv, 1, len(rows), Hq, Hk, 1e-6, 1e4, *b, pos=pos,
                                   cos_tab=ct, sin_tab=st)
    flat = lambda t: t.reshape(B * S, *t.shape[2:])[rows]
    assert oracle.rel_err(host(flat(q)), want[0][0]) <= TOL["bf16"]
    assert oracle.rel_err(host(flat(k)), want[1][0]) <= TOL["bf16"]
    assert oracle.rel_err(host(flat(v)), want[2][0]) <= TOL["bf16"]
    assert oracle.rel_err(host(rstd[rows]), want[3]) <= TOL["f32"]
