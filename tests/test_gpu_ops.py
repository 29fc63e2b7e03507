"""GPU parity of RMSNorm, RoPE and SwiGLU against the fp64 oracle, through
the C-ABI (libliger.so), element by element.

Sizes: the tiny decoder-op set (fp32 and bf16), ragged medium cases that
span many blocks and end in a partial vector / row group, and the full
Llama-3-8B / SwiGLU shapes in the launch configuration the benchmark times,
checked on sampled rows (and in full where the oracle is cheap)."""
import numpy as np
import pytest

import datagen
import oracle
from datagen import workloads
from gpu_util import TOL, bits, dev, host, storage

pytestmark = pytest.mark.gpu


def _rms(cuda_lib, x, w, eps):
    import torch
    tx, tw = dev(x), dev(w)
    y = torch.empty_like(tx)
    rstd = torch.empty(x.size // x.shape[-1], dtype=torch.float32, device="cuda")
    cuda_lib.liger_rmsnorm_fwd(tx, tw, y, rstd, eps)
    return tx, tw, y, rstd


# ---------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rmsnorm_tiny(cuda_lib, dtype):
    r = workloads.tiny(dtype)["rmsnorm"]
    x, w, dy = r.make("x"), r.make("w"), r.make("dy")
    eps = r.params["eps"]
    tx, tw, y, rstd = _rms(cuda_lib, x, w, eps)
    oy, orstd = oracle.rmsnorm_fwd(x, w, eps)
    assert oracle.rel_err(host(y), oy) <= TOL[dtype]
    assert oracle.rel_err(host(rstd), orstd) <= 1e-5
    import torch
    ws = torch.empty(cuda_lib.liger_rmsnorm_bwd_workspace(*x.shape), dtype=torch.uint8, device="cuda")
    dx, dw = torch.empty_like(tx), torch.empty_like(tw)
    cuda_lib.liger_rmsnorm_bwd(dev(dy), tx, tw, rstd, dx, dw, ws)
    odx, odw = oracle.rmsnorm_bwd(dy, x, w, eps)
    assert oracle.rel_err(host(dx), odx) <= TOL[dtype]
    assert oracle.rel_err(host(dw), odw) <= TOL[dtype]


@pytest.mark.parametrize("dtype,rows,cols", [("bf16", 1237, 4096), ("f32", 1003, 4096), ("bf16", 517, 8192),
                                             ("bf16", 77, 1000), ("f32", 33, 1001), ("bf16", 64, 16384),
                                             ("bf16", 5, 8)])
def test_rmsnorm_ragged(cuda_lib, dtype, rows, cols):
    import torch
    x = datagen.normal(11, "rx", (rows, cols), dtype)
    w = datagen.normal(11, "rw", (cols,), dtype, 1.0, 0.1)
    dy = datagen.normal(11, "rdy", (rows, cols), dtype)
    tx, tw, y, rstd = _rms(cuda_lib, x, w, 1e-5)
    oy, _ = oracle.rmsnorm_fwd(x, w, 1e-5)
    assert oracle.rel_err(host(y), oy) <= TOL[dtype]
    ws = torch.empty(cuda_lib.liger_rmsnorm_bwd_workspace(rows, cols), dtype=torch.uint8, device="cuda")
    dx, dw = torch.empty_like(tx), torch.empty_like(tw)
    cuda_lib.liger_rmsnorm_bwd(dev(dy), tx, tw, rstd, dx, dw, ws)
    odx, odw = oracle.rmsnorm_bwd(dy, x, w, 1e-5)
    assert oracle.rel_err(host(dx), odx) <= TOL[dtype]
    assert oracle.rel_err(host(dw), odw) <= TOL[dtype]


def test_rmsnorm_llama3_full_size(cuda_lib):
    """x [4*8192, 4096] bf16, eps 1e-5: sampled rows of y / dx, all of dw."""
    import torch
    r = workloads.rmsnorm_rope_llama3()["rmsnorm"]
    x, w, dy = r.make("x"), r.make("w"), r.make("dy")
    eps = r.params["eps"]
    tx, tw, y, rstd = _rms(cuda_lib, x, w, eps)
    ws = torch.empty(cuda_lib.liger_rmsnorm_bwd_workspace(*x.shape), dtype=torch.uint8, device="cuda")
    dx, dw = torch.empty_like(tx), torch.empty_like(tw)
    cuda_lib.liger_rmsnorm_bwd(dev(dy), tx, tw, rstd, dx, dw, ws)
    rows = np.random.default_rng(2).choice(x.shape[0], 256, replace=False)
    rows = np.concatenate([[0, x.shape[0] - 1], rows])
    oy, _ = oracle.rmsnorm_fwd(x[rows], w, eps)
    odx, _ = oracle.rmsnorm_bwd(dy[rows], x[rows], w, eps)
    assert oracle.rel_err(host(y)[rows], oy) <= 2e-2
    assert oracle.rel_err(host(dx)[rows], odx) <= 2e-2
    _, odw = oracle.rmsnorm_bwd(dy, x, w, eps)
    assert oracle.rel_err(host(dw), odw) <= 2e-2


def test_rmsnorm_deterministic_dw(cuda_lib):
    import torch
    x = datagen.normal(5, "dx", (3000, 4096), "bf16")
    w = datagen.normal(5, "dw", (4096,), "bf16", 1.0, 0.1)
    dy = datagen.normal(5, "ddy", (3000, 4096), "bf16")
    tx, tw, y, rstd = _rms(cuda_lib, x, w, 1e-6)
    ws = torch.empty(cuda_lib.liger_rmsnorm_bwd_workspace(3000, 4096), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        dx, dw = torch.empty_like(tx), torch.empty_like(tw)
        cuda_lib.liger_rmsnorm_bwd(dev(dy), tx, tw, rstd, dx, dw, ws)
        outs.append((bits(dx), bits(dw)))
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1])


# -------------------------------------------------------------------- RoPE
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rope_tiny(cuda_lib, dtype):
    p = workloads.tiny(dtype)["rope"]
    theta = p.params["theta"]
    q, k, dq, dk = p.make("q"), p.make("k"), p.make("dq"), p.make("dk")
    tq, tk = dev(q), dev(k)
    cuda_lib.liger_rope_fwd(tq, tk, None, theta)
    assert oracle.rel_err(host(tq), oracle.rope(q, theta)) <= TOL[dtype]
    assert oracle.rel_err(host(tk), oracle.rope(k, theta)) <= TOL[dtype]
    tdq, tdk = dev(dq), dev(dk)
    cuda_lib.liger_rope_bwd(tdq, tdk, None, theta)
    assert oracle.rel_err(host(tdq), oracle.rope(dq, theta, sign=-1)) <= TOL[dtype]
    assert oracle.rel_err(host(tdk), oracle.rope(dk, theta, sign=-1)) <= TOL[dtype]


@pytest.mark.parametrize("dtype,B,S,Hq,Hk,D", [("f32", 3, 37, 5, 2, 128), ("bf16", 2, 300, 7, 3, 64),
                                              ("f32", 1, 9, 3, 1, 6), ("bf16", 11, 5, 2, 2, 24)])
def test_rope_ragged_positions(cuda_lib, dtype, B, S, Hq, Hk, D):
    """Explicit positions (large, per batch row), odd head counts, head_dim
    without a full vector (scalar path), batch beyond one batch group."""
    q = datagen.normal(3, "pq", (B, S, Hq, D), dtype)
    k = datagen.normal(3, "pk", (B, S, Hk, D), dtype)
    pos = datagen.positions(3, "pp", (B, S), 32768)
    tq, tk = dev(q), dev(k)
    cuda_lib.liger_rope_fwd(tq, tk, dev(pos), 5e5)
    assert oracle.rel_err(host(tq), oracle.rope(q, 5e5, pos=pos)) <= TOL[dtype]
    assert oracle.rel_err(host(tk), oracle.rope(k, 5e5, pos=pos)) <= TOL[dtype]
    cuda_lib.liger_rope_bwd(tq, tk, dev(pos), 5e5)
    q64 = datagen.to_f64(q, dtype)
    assert oracle.rel_err(host(tq), q64) <= (1e-5 if dtype == "f32" else 2e-2)


@pytest.mark.parametrize("dtype,B,S,Hq,Hk,D", [("f32", 1, 40, 400, 112, 128),    # a token row of 256 KB: no staged tile
                                               ("bf16", 70000, 2, 1, 1, 64)])    # batch beyond the staged grid
def test_rope_fallback_layouts(cuda_lib, dtype, B, S, Hq, Hk, D):
    """The RoPE forms the staged kernel does not take: token rows larger than a
    block's shared memory, and batches beyond its grid; explicit positions."""
    q = datagen.normal(4, "fq", (B, S, Hq, D), dtype)
    k = datagen.normal(4, "fk", (B, S, Hk, D), dtype)
    pos = datagen.positions(4, "fp", (B, S), 8192)
    tq, tk = dev(q), dev(k)
    cuda_lib.liger_rope_fwd(tq, tk, dev(pos), 1e4)
    assert oracle.rel_err(host(tq), oracle.rope(q, 1e4, pos=pos)) <= TOL[dtype]
    assert oracle.rel_err(host(tk), oracle.rope(k, 1e4, pos=pos)) <= TOL[dtype]
    cuda_lib.liger_rope_bwd(tq, tk, dev(pos), 1e4)
    assert oracle.rel_err(host(tq), datagen.to_f64(q, dtype)) <= (1e-5 if dtype == "f32" else 2e-2)


def test_rope_fp32_long_positions_accuracy(cuda_lib):
    """fp32 at positions up to 32767: the fp64 angle reduction keeps ~1e-6."""
    q = datagen.normal(9, "lq", (1, 4, 2, 128), "f32")
    pos = np.array([[0, 8191, 16384, 32767]], np.int32)
    tq = dev(q)
    cuda_lib.liger_rope_fwd(tq, None, dev(pos), 5e5)
    assert oracle.rel_err(host(tq), oracle.rope(q, 5e5, pos=pos)) <= 1e-5


def test_rope_llama3_full_size(cuda_lib):
    """Q [4, 8192, 32, 128], K [4, 8192, 8, 128] bf16, theta 5e5: sampled positions."""
    p = workloads.rmsnorm_rope_llama3()["rope"]
    theta = p.params["theta"]
    q, k = p.make("q"), p.make("k")
    tq, tk = dev(q), dev(k)
    cuda_lib.liger_rope_fwd(tq, tk, None, theta)
    hq, hk = host(tq), host(tk)
    ss = np.concatenate([[0, 1, 8191], np.random.default_rng(0).choice(8192, 61, replace=False)])
    for b in range(4):
        pos = np.tile(ss.astype(np.int32), (1, 1))
        oq = oracle.rope(np.ascontiguousarray(q[b:b + 1, ss]), theta, pos=pos)
        ok = oracle.rope(np.ascontiguousarray(k[b:b + 1, ss]), theta, pos=pos)
        assert oracle.rel_err(hq[b:b + 1, ss], oq) <= 2e-2
        assert oracle.rel_err(hk[b:b + 1, ss], ok) <= 2e-2


def test_rope_bwd_llama3_full_size(cuda_lib):
    """The backward at the same shape: dQ [4, 8192, 32, 128], dK [4, 8192, 8, 128]
    bf16 rotated by -phi in place, theta 5e5: sampled positions of every batch
    row against the oracle's rotation with sign -1."""
    p = workloads.rmsnorm_rope_llama3()["rope"]
    theta = p.params["theta"]
    dq, dk = p.make("dq"), p.make("dk")
    tq, tk = dev(dq), dev(dk)
    cuda_lib.liger_rope_bwd(tq, tk, None, theta)
    hq, hk = host(tq), host(tk)
    ss = np.concatenate([[0, 1, 4095, 8191], np.random.default_rng(1).choice(8192, 60, replace=False)])
    pos = ss.astype(np.int32)[None, :]
    for b in range(4):
        oq = oracle.rope(np.ascontiguousarray(dq[b:b + 1, ss]), theta, sign=-1, pos=pos)
        ok = oracle.rope(np.ascontiguousarray(dk[b:b + 1, ss]), theta, sign=-1, pos=pos)
        assert oracle.rel_err(hq[b:b + 1, ss], oq) <= 2e-2
        assert oracle.rel_err(hk[b:b + 1, ss], ok) <= 2e-2


# ------------------------------------------------------------------ SwiGLU
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_swiglu_tiny(cuda_lib, dtype):
    import torch
    s = workloads.tiny(dtype)["swiglu"]
    g, u, dy = s.make("gate"), s.make("up"), s.make("dy")
    tg, tu = dev(g), dev(u)
    y = torch.empty_like(tg)
    cuda_lib.liger_swiglu_fwd(tg, tu, y)
    assert oracle.rel_err(host(y), oracle.swiglu_fwd(g, u)) <= TOL[dtype]
    dg, du = torch.empty_like(tg), torch.empty_like(tu)
    cuda_lib.liger_swiglu_bwd(dev(dy), tg, tu, dg, du)
    odg, odu = oracle.swiglu_bwd(dy, g, u)
    assert oracle.rel_err(host(dg), odg) <= TOL[dtype]
    assert oracle.rel_err(host(du), odu) <= TOL[dtype]


@pytest.mark.parametrize("dtype,n", [("bf16", 1_000_003), ("f32", 999_999), ("bf16", 7), ("f32", 3)])
def test_swiglu_ragged_inplace(cuda_lib, dtype, n):
    g = datagen.normal(4, "sg", (n,), dtype, 0.0, 3.0)
    u = datagen.normal(4, "su", (n,), dtype)
    dy = datagen.normal(4, "sd", (n,), dtype)
    tg, tu = dev(g), dev(u)
    y = dev(g)                                 # y aliases a copy of gate
    cuda_lib.liger_swiglu_fwd(y, tu, y)
    assert oracle.rel_err(host(y), oracle.swiglu_fwd(g, u)) <= TOL[dtype]
    cuda_lib.liger_swiglu_bwd(dev(dy), tg, tu, tg, tu)   # in place: dgate -> gate, dup -> up
    odg, odu = oracle.swiglu_bwd(dy, g, u)
    assert oracle.rel_err(host(tg), odg) <= TOL[dtype]
    assert oracle.rel_err(host(tu), odu) <= TOL[dtype]


def test_swiglu_llama_full_size(cuda_lib):
    """gate/up [4, 2048, 11008] bf16: full comparison (the oracle takes seconds)."""
    import torch
    s = workloads.swiglu_llama()
    g, u, dy = s.make("gate"), s.make("up"), s.make("dy")
    tg, tu = dev(g), dev(u)
    y = torch.empty_like(tg)
    cuda_lib.liger_swiglu_fwd(tg, tu, y)
    sl = slice(0, None, 7)
    gf, uf, dyf = g.reshape(-1)[sl], u.reshape(-1)[sl], dy.reshape(-1)[sl]
    assert oracle.rel_err(host(y).reshape(-1)[sl], oracle.swiglu_fwd(gf, uf)) <= 2e-2
    dg, du = torch.empty_like(tg), torch.empty_like(tu)
    cuda_lib.liger_swiglu_bwd(dev(dy), tg, tu, dg, du)
    odg, odu = oracle.swiglu_bwd(dyf, gf, uf)
    assert oracle.rel_err(host(dg).reshape(-1)[sl], odg) <= 2e-2
    assert oracle.rel_err(host(du).reshape(-1)[sl], odu) <= 2e-2


# --------------------------------------------------------------- edge cases
def test_zero_sized_calls(cuda_lib):
    import torch
    e = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    cuda_lib.liger_rmsnorm_fwd(e, w, e, None, 1e-6)
    cuda_lib.liger_swiglu_fwd(e, e, e)
    q = torch.empty(2, 0, 4, 64, dtype=torch.bfloat16, device="cuda")
    cuda_lib.liger_rope_fwd(q, q, None, 1e4)
    dw = torch.full((64,), 3.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.liger_rmsnorm_bwd(e, e, w, torch.empty(0, device="cuda"), e, dw, None)
    assert torch.all(dw == 0)


# ------------------------------------------------------------ RoPE variants
@pytest.mark.parametrize("dtype,pairing,D", [("bf16", "interleaved", 128), ("f32", "interleaved", 64),
                                             ("bf16", "half", 128), ("f32", "interleaved", 6),
                                             ("bf16", "interleaved", 24)])
def test_rope_ex_packed_qkv_views(cuda_lib, dtype, pairing, D):
    """q and k as views into a packed [B, S, (Hq + 2 Hk) * D] QKV buffer; v untouched."""
    import torch
    B, S, Hq, Hk = 2, 37, 5, 2
    W = (Hq + 2 * Hk) * D
    qkv = datagen.normal(41, "qkv", (B, S, W), dtype)
    pos = datagen.positions(41, "qp", (B, S), 32768)
    t = dev(qkv)
    tq = t.view(-1)[0:]                              # q starts at element 0 of each token
    tk = t.view(-1)[Hq * D:]                         # k starts after the q heads
    cuda_lib.liger_rope_fwd_ex(tq, tk, W, W, Hq, Hk, D, B, S, dev(pos), 5e5, pairing)
    out = host(t)
    q = np.ascontiguousarray(qkv[:, :, : Hq * D].reshape(B, S, Hq, D))
    k = np.ascontiguousarray(qkv[:, :, Hq * D: (Hq + Hk) * D].reshape(B, S, Hk, D))
    oq = oracle.rope_ex(q, 5e5, pos=pos, pairing=pairing).reshape(B, S, Hq * D)
    ok = oracle.rope_ex(k, 5e5, pos=pos, pairing=pairing).reshape(B, S, Hk * D)
    assert oracle.rel_err(out[:, :, : Hq * D], oq) <= TOL[dtype]
    assert oracle.rel_err(out[:, :, Hq * D: (Hq + Hk) * D], ok) <= TOL[dtype]
    assert np.array_equal(bits(t)[:, :, (Hq + Hk) * D:], qkv[:, :, (Hq + Hk) * D:].view(bits(t).dtype))
    cuda_lib.liger_rope_bwd_ex(tq, tk, W, W, Hq, Hk, D, B, S, dev(pos), 5e5, pairing)
    assert oracle.rel_err(host(t), datagen.to_f64(qkv, dtype)) <= (1e-5 if dtype == "f32" else 2e-2)
    del torch


@pytest.mark.parametrize("pairing", ["half", "interleaved"])
def test_rope_ex_explicit_tables(cuda_lib, pairing):
    """Caller-supplied cos/sin tables (a scaled schedule: angles p * 0.25 * theta^(-2i/D))."""
    import torch
    B, S, H, D = 1, 64, 3, 64
    i = np.arange(D // 2)
    ang = np.arange(S)[:, None] * 0.25 * (1e4 ** (-2.0 * i / D))[None, :]
    cos_t, sin_t = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    q = datagen.normal(42, "tq", (B, S, H, D), "f32")
    tq = dev(q)
    cuda_lib.liger_rope_fwd_ex(tq, None, H * D, 0, H, 0, D, B, S, None, 0.0, pairing,
                               torch.from_numpy(cos_t).cuda(), torch.from_numpy(sin_t).cuda())
    want = oracle.rope_ex(q, 0.0, pairing=pairing, cos_tab=cos_t.astype(np.float64), sin_tab=sin_t.astype(np.float64))
    assert oracle.rel_err(host(tq), want) <= 1e-5
