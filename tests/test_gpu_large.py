"""Maximum sizes: SwiGLU, RMSNorm and RoPE on tensors of more than 2^31
elements, where any 32-bit element offset would wrap.

Each input is a seeded period of the generator (a length prime to the row
width, so rows differ) repeated on the device to the full size; the oracle
then knows every element (element i is period[i mod P]) and is evaluated on
sampled elements, rows or positions: the first ones, those on both sides of
the 2^31 element boundary, the ragged tail, and random ones."""
import numpy as np
import pytest

import datagen
import oracle
from gpu_util import dev, host

pytestmark = pytest.mark.gpu

BIG = (1 << 31) + 24        # elements: past 2^31, and not a whole number of 16-byte vectors


def _tiled(seed, name, period, total, mean=0.0, std=1.0):
    base = datagen.normal(seed, name, (period,), "bf16", mean, std)
    t = dev(base)
    return base, t.repeat(-(-total // period))[:total].contiguous()


def _at(base, idx):
    return base[np.asarray(idx, np.int64) % base.size]


def _sample(n, unit=1, k=64, seed=0):
    """Indices (in units of `unit` elements) at the start, around 2^31 elements, at the end, random."""
    m = n // unit
    b = (1 << 31) // unit
    s = np.concatenate([np.arange(4), np.arange(b - 3, b + 3), np.arange(m - 4, m),
                        np.random.default_rng(seed).choice(m, k, replace=False)])
    return np.unique(s[(s >= 0) & (s < m)])


def test_swiglu_past_2_31_elements(cuda_lib):
    import torch
    P = 1_000_003
    gb, g = _tiled(61, "bg", P, BIG)
    ub, u = _tiled(61, "bu", P, BIG)
    y = torch.empty_like(g)
    cuda_lib.liger_swiglu_fwd(g, u, y)
    idx = _sample(BIG, k=256)
    ti = torch.as_tensor(idx, device="cuda")
    assert oracle.rel_err(host(y[ti]), oracle.swiglu_fwd(_at(gb, idx), _at(ub, idx))) <= 2e-2
    del y
    db, d = _tiled(61, "bdy", P, BIG)
    dg, du = torch.empty_like(g), torch.empty_like(g)
    cuda_lib.liger_swiglu_bwd(d, g, u, dg, du)
    odg, odu = oracle.swiglu_bwd(_at(db, idx), _at(gb, idx), _at(ub, idx))
    assert oracle.rel_err(host(dg[ti]), odg) <= 2e-2
    assert oracle.rel_err(host(du[ti]), odu) <= 2e-2


def test_rmsnorm_past_2_31_elements(cuda_lib):
    import torch
    H = 4096
    rows = (1 << 31) // H + 8
    P = 4096 * 67 + 8
    xb, x = _tiled(62, "bx", P, rows * H)
    wb = datagen.normal(62, "bw", (H,), "bf16", 1.0, 0.1)
    w = dev(wb)
    x = x.view(rows, H)
    y = torch.empty_like(x)
    rstd = torch.empty(rows, dtype=torch.float32, device="cuda")
    cuda_lib.liger_rmsnorm_fwd(x, w, y, rstd, 1e-5)
    rs = _sample(rows * H, unit=H, k=24)
    rows_x = np.stack([_at(xb, np.arange(r * H, (r + 1) * H)) for r in rs])
    oy, orstd = oracle.rmsnorm_fwd(rows_x, wb, 1e-5)
    ti = torch.as_tensor(rs, device="cuda")
    assert oracle.rel_err(host(y[ti]), oy) <= 2e-2
    assert oracle.rel_err(host(rstd[ti]), orstd) <= 1e-5
    del y
    db, d = _tiled(62, "bdy", P, rows * H)
    d = d.view(rows, H)
    dx, dw = torch.empty_like(x), torch.empty_like(w)
    ws = torch.empty(cuda_lib.liger_rmsnorm_bwd_workspace(rows, H), dtype=torch.uint8, device="cuda")
    cuda_lib.liger_rmsnorm_bwd(d, x, w, rstd, dx, dw, ws)
    rows_d = np.stack([_at(db, np.arange(r * H, (r + 1) * H)) for r in rs])
    odx, _ = oracle.rmsnorm_bwd(rows_d, rows_x, wb, 1e-5)
    assert oracle.rel_err(host(dx[ti]), odx) <= 2e-2
    assert bool(torch.isfinite(dw.float()).all())


def test_rope_past_2_31_elements(cuda_lib):
    import torch
    S, NH, D = (1 << 31) // (32 * 128) + 8, 32, 128
    P = 32 * 128 * 53 + 16
    qb, q = _tiled(63, "bq", P, S * NH * D)
    q = q.view(1, S, NH, D)
    cuda_lib.liger_rope_fwd(q, None, None, 5e5)
    ps = _sample(S * NH * D, unit=NH * D, k=24)
    tok = np.stack([_at(qb, np.arange(p * NH * D, (p + 1) * NH * D)).reshape(NH, D) for p in ps])[None]
    oq = oracle.rope(np.ascontiguousarray(tok), 5e5, pos=ps.astype(np.int32)[None])
    assert oracle.rel_err(host(q[0, torch.as_tensor(ps, device="cuda")])[None], oq) <= 2e-2
