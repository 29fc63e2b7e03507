"""Pins of the fp64 oracle to facts other than itself.

Each operator is checked against closed forms, hand-worked values (tests/
golden), invariants of the mathematics, and central finite differences on
tiny inputs, chosen so that a plausible slip (a dropped term, a wrong sign,
index or pairing, a transposed operand, eps in the wrong place, sum instead
of mean) fails at least one test.
"""
import math

import numpy as np
import pytest

import oracle
from conftest import golden

RNG = np.random.default_rng(12345)


# ------------------------------------------------------------------ RMSNorm
def test_rmsnorm_constant_row_closed_form():
    g = golden("rmsnorm_closed_forms.json")
    x = np.full((2, g["H"]), g["a"]); w = np.ones(g["H"])
    y, rstd = oracle.rmsnorm_fwd(x, w, g["eps"])
    assert np.allclose(y, g["y"], rtol=1e-15, atol=0)
    assert np.allclose(rstd, g["rstd"], rtol=1e-15, atol=0)


def test_rmsnorm_scale_invariance_eps0():
    x = RNG.standard_normal((5, 37)); w = 1 + 0.1 * RNG.standard_normal(37)
    y0, _ = oracle.rmsnorm_fwd(x, w, 0.0)
    for c in (0.5, 3.0, 1e3):
        yc, _ = oracle.rmsnorm_fwd(c * x, w, 0.0)
        assert np.max(np.abs(yc - y0)) < 1e-13


def test_rmsnorm_unit_mean_square_and_weight_per_feature():
    x = RNG.standard_normal((4, 64))
    y, _ = oracle.rmsnorm_fwd(x, np.ones(64), 0.0)
    assert np.allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)   # mean, not sum
    w = np.arange(1, 9, dtype=np.float64)
    y, _ = oracle.rmsnorm_fwd(np.full((1, 8), -3.0), w, 0.0)
    assert np.allclose(y[0], -w, rtol=1e-15)                      # plain x*r*w, not (1+w)


def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        xp = x.copy(); xm = x.copy(); xp[i] += h; xm[i] -= h
        g[i] = (f(xp) - f(xm)) / (2 * h)
    return g


def test_rmsnorm_bwd_finite_differences():
    rows, H, eps = 3, 7, 1e-3
    x = RNG.standard_normal((rows, H)); w = 1 + 0.1 * RNG.standard_normal(H); dy = RNG.standard_normal((rows, H))
    dx, dw = oracle.rmsnorm_bwd(dy, x, w, eps)
    L = lambda xx: float(np.sum(dy * oracle.rmsnorm_fwd(xx, w, eps)[0]))
    Lw = lambda ww: float(np.sum(dy * oracle.rmsnorm_fwd(x, ww, eps)[0]))
    fx, fw = _fd(L, x), _fd(Lw, w)
    assert np.max(np.abs(dx - fx)) / np.max(np.abs(fx)) < 1e-7
    assert np.max(np.abs(dw - fw)) / np.max(np.abs(fw)) < 1e-7


def test_rmsnorm_bwd_orthogonal_to_x_when_eps0():
    x = RNG.standard_normal((6, 33)); w = 1 + 0.1 * RNG.standard_normal(33); dy = RNG.standard_normal((6, 33))
    dx, _ = oracle.rmsnorm_bwd(dy, x, w, 0.0)
    assert np.max(np.abs(np.sum(dx * x, axis=1))) < 1e-12


# --------------------------------------------------------------------- RoPE
def test_rope_single_feature_angles():
    for c in golden("rope_angles.json")["cases"]:
        D, i, p = c["D"], c["i"], c["p"]
        t = np.zeros((1, p + 1, 1, D)); t[0, p, 0, i] = 1.0
        out = oracle.rope(t, c["theta"])
        assert abs(out[0, p, 0, i] - c["cos"]) < 1e-12
        assert abs(out[0, p, 0, i + D // 2] - c["sin"]) < 1e-12
        others = np.delete(out[0, p, 0], [i, i + D // 2])
        assert np.all(others == 0)
        # the second half of a pair rotates the other way round
        t2 = np.zeros_like(t); t2[0, p, 0, i + D // 2] = 1.0
        o2 = oracle.rope(t2, c["theta"])
        assert abs(o2[0, p, 0, i] + c["sin"]) < 1e-12 and abs(o2[0, p, 0, i + D // 2] - c["cos"]) < 1e-12


def test_rope_norm_identity_inverse():
    t = RNG.standard_normal((2, 9, 3, 16))
    out = oracle.rope(t, 1e4)
    half = 8
    n_in = t[..., :half] ** 2 + t[..., half:] ** 2
    n_out = out[..., :half] ** 2 + out[..., half:] ** 2
    assert np.max(np.abs(n_in - n_out)) < 1e-13
    assert np.array_equal(out[:, 0], t[:, 0])                     # position 0: identity
    back = oracle.rope(out, 1e4, sign=-1)
    assert np.max(np.abs(back - t)) < 1e-13                        # bwd o fwd = identity


def test_rope_relative_position():
    q = RNG.standard_normal((1, 1, 1, 32)); k = RNG.standard_normal((1, 1, 1, 32))
    def dot(m, n):
        rq = oracle.rope(q, 5e5, pos=np.array([[m]], np.int32))
        rk = oracle.rope(k, 5e5, pos=np.array([[n]], np.int32))
        return float(np.sum(rq * rk))
    for m, n in ((5, 2), (100, 40), (8000, 7999)):
        assert abs(dot(m, n) - dot(m + 17, n + 17)) < 1e-10
    assert abs(dot(5, 2) - dot(9, 2)) > 1e-3


def test_rope_bwd_is_adjoint():
    x = RNG.standard_normal((2, 5, 2, 8)); dy = RNG.standard_normal((2, 5, 2, 8))
    pos = np.array([[3, 1, 4, 1, 5], [9, 2, 6, 5, 3]], np.int32)
    lhs = np.sum(dy * oracle.rope(x, 1e4, pos=pos))
    rhs = np.sum(oracle.rope(dy, 1e4, sign=-1, pos=pos) * x)
    assert abs(lhs - rhs) < 1e-12


# ------------------------------------------------------------------- SwiGLU
def test_swiglu_values():
    g = golden("silu_values.json")
    gate = np.array([0.0, 1.0, -1.0, 40.0, -40.0]); up = np.array([2.0, 3.0, 5.0, 0.5, 7.0])
    y = oracle.swiglu_fwd(gate, up)
    assert y[0] == 0.0
    assert abs(y[1] - 3 * g["silu_1"]) < 1e-15 and abs(y[2] - 5 * g["silu_m1"]) < 1e-15
    assert abs(y[3] - 40 * 0.5) < 1e-12
    assert abs(y[4] - (-280.0 * math.exp(-40) / (1 + math.exp(-40)))) < 1e-28   # -40 * sigmoid(-40) * 7
    dy = np.array([1.5, 2.0, 1.0, 1.0, 1.0])
    dg, du = oracle.swiglu_bwd(dy, gate, up)
    assert abs(dg[0] - 1.5 * 2.0 * g["dsilu_0"]) < 1e-15 and du[0] == 0.0
    assert abs(dg[1] - 2.0 * 3.0 * g["dsilu_1"]) < 1e-14
    assert abs(du[1] - 2.0 * g["silu_1"]) < 1e-15


def test_swiglu_bwd_finite_differences():
    gate = RNG.standard_normal(11) * 2; up = RNG.standard_normal(11); dy = RNG.standard_normal(11)
    dg, du = oracle.swiglu_bwd(dy, gate, up)
    fg = _fd(lambda gg: float(np.sum(dy * oracle.swiglu_fwd(gg, up))), gate)
    fu = _fd(lambda uu: float(np.sum(dy * oracle.swiglu_fwd(gate, uu))), up)
    assert np.max(np.abs(dg - fg)) < 1e-8 and np.max(np.abs(du - fu)) < 1e-8


# --------------------------------------------------------------- linear CE
def test_ce_three_class_golden():
    g = golden("ce_three_class.json")
    X = np.array([g["logits"]]); W = np.eye(3)
    r = oracle.linear_ce(X, W, np.array([g["label"]]))
    assert abs(r["loss"] - g["loss"]) < 1e-14
    assert np.max(np.abs(r["dX"][0] - np.array(g["grad"]))) < 1e-15   # W = I: dX = D
    assert np.max(np.abs(r["dW"] - np.outer(g["grad"], g["logits"]))) < 1e-14


@pytest.mark.parametrize("V", [1024, 5, 77])
def test_ce_uniform_logits_is_ln_v(V):
    T, H = 6, 4
    X = RNG.standard_normal((T, H)); W = np.zeros((V, H))
    lab = RNG.integers(0, V, T)
    assert abs(oracle.linear_ce(X, W, lab)["loss"] - math.log(V)) < 1e-13
    W2 = RNG.standard_normal((V, H))
    assert abs(oracle.linear_ce(np.zeros((T, H)), W2, lab)["loss"] - math.log(V)) < 1e-13


def test_ce_large_vocab_ln_v():
    for V in (128256, 151936):
        r = oracle.linear_ce(np.zeros((1, 2)), np.ones((V, 2)), np.array([V - 1]), want_grads=False)
        assert abs(r["loss"] - math.log(V)) < 1e-12


def test_ce_grad_rows_sum_zero_and_ignore():
    T, H, V = 7, 5, 9
    X = RNG.standard_normal((T, H)); W = RNG.standard_normal((V, H))
    lab = RNG.integers(0, V, T); lab[[1, 4]] = -100
    r = oracle.linear_ce(X, W, lab)
    # sum over the vocabulary of dW rows = sum_t (sum_v D_tv) X_t = 0
    assert np.max(np.abs(r["dW"].sum(axis=0))) < 1e-14
    assert np.all(r["dX"][[1, 4]] == 0.0)
    X2 = X.copy(); X2[[1, 4]] = 1e3                                  # ignored rows do not matter
    r2 = oracle.linear_ce(X2, W, lab)
    assert abs(r2["loss"] - r["loss"]) < 1e-14 and np.max(np.abs(r2["dW"] - r["dW"])) < 1e-14


def test_ce_all_ignored_and_bad_label():
    X = RNG.standard_normal((3, 2)); W = RNG.standard_normal((4, 2))
    r = oracle.linear_ce(X, W, np.array([-100, -100, -100]))
    assert r["loss"] == 0.0 and np.all(r["dX"] == 0) and np.all(r["dW"] == 0)
    with pytest.raises(ValueError, match="-5"):
        oracle.linear_ce(X, W, np.array([0, 4, 1]))


def test_ce_finite_differences_mean_and_sum():
    T, H, V = 4, 3, 5
    X = RNG.standard_normal((T, H)); W = RNG.standard_normal((V, H)); lab = np.array([2, -100, 4, 0])
    for red in ("mean", "sum"):
        r = oracle.linear_ce(X, W, lab, reduction=red, grad_scale=1.7)
        fX = _fd(lambda xx: 1.7 * oracle.linear_ce(xx, W, lab, reduction=red, want_grads=False)["loss"], X)
        fW = _fd(lambda ww: 1.7 * oracle.linear_ce(X, ww, lab, reduction=red, want_grads=False)["loss"], W)
        assert np.max(np.abs(r["dX"] - fX)) < 1e-8
        assert np.max(np.abs(r["dW"] - fW)) < 1e-8
    rm = oracle.linear_ce(X, W, lab)["loss"]; rs = oracle.linear_ce(X, W, lab, reduction="sum")["loss"]
    assert abs(rs - 3 * rm) < 1e-13                                   # 3 valid rows


def test_ce_rows_matches_full_definition():
    T, H, V = 9, 6, 13
    X = RNG.standard_normal((T, H)); W = RNG.standard_normal((V, H)); lab = RNG.integers(0, V, T); lab[2] = -100
    full = oracle.linear_ce(X, W, lab)
    rows = np.array([0, 2, 8, 5])
    part = oracle.linear_ce_rows(X, W, lab, rows)
    assert np.max(np.abs(part["dX"] - full["dX"][rows])) < 1e-15
    assert np.max(np.abs(part["lse"] - full["lse"][rows])) < 1e-15
    assert abs(part["loss_term"][1]) == 0.0


def test_ce_rows_fwd_and_dw_rows_match_full_definition():
    T, H, V = 11, 5, 17
    X = RNG.standard_normal((T, H)); W = RNG.standard_normal((V, H)); lab = RNG.integers(0, V, T)
    lab[3] = -100; lab[7] = lab[0]                        # an ignored row, a label shared by two tokens
    for red, gs in (("mean", 1.0), ("sum", 0.3)):
        full = oracle.linear_ce(X, W, lab, reduction=red, grad_scale=gs)
        fw = oracle.linear_ce_rows_fwd(X, W, lab, np.arange(T))
        assert np.max(np.abs(fw["lse"] - full["lse"])) < 1e-15
        valid = lab != -100
        n = valid.sum() if red == "mean" else 1
        assert abs(fw["loss_term"].sum() / n - full["loss"]) < 1e-14
        vrows = np.array([lab[0], 0, V - 1, 9])
        dw = oracle.linear_ce_dw_rows(X, W, lab, full["lse"], vrows, reduction=red, grad_scale=gs)
        assert np.max(np.abs(dw - full["dW"][vrows])) < 1e-14


def test_storage_widening_is_exact():
    import datagen
    b = datagen.normal(0, "w", (4, 8), "bf16"); f = datagen.bf16_bits_to_f32(b)
    y1, _ = oracle.rmsnorm_fwd(b, datagen.f32_to_bf16_bits(np.ones(8, np.float32)), 1e-6)
    y2, _ = oracle.rmsnorm_fwd(f.astype(np.float64), np.ones(8), 1e-6)
    assert np.array_equal(y1, y2)


# ------------------------------------------------------------ RoPE variants
def test_rope_ex_half_pairing_equals_rope():
    t = RNG.standard_normal((2, 7, 3, 16))
    pos = RNG.integers(0, 5000, (2, 7)).astype(np.int32)
    assert np.array_equal(oracle.rope_ex(t, 5e5, pos=pos), oracle.rope(t, 5e5, pos=pos))


def test_rope_ex_interleaved_single_feature_angles():
    # interleaved pairs (2i, 2i+1): a unit vector at feature 2i rotates to (cos, sin) at (2i, 2i+1)
    for c in golden("rope_angles.json")["cases"]:
        D, i, p = c["D"], c["i"], c["p"]
        t = np.zeros((1, p + 1, 1, D)); t[0, p, 0, 2 * i] = 1.0
        out = oracle.rope_ex(t, c["theta"], pairing="interleaved")
        assert abs(out[0, p, 0, 2 * i] - c["cos"]) < 1e-12 and abs(out[0, p, 0, 2 * i + 1] - c["sin"]) < 1e-12
        assert np.count_nonzero(np.abs(out[0, p, 0]) > 1e-15) == 2


def test_rope_ex_table_matches_schedule_and_inverse():
    D, P = 16, 40
    i = np.arange(D // 2)
    ang = np.arange(P)[:, None] * (1e4 ** (-2.0 * i / D))[None, :]
    cos_t, sin_t = np.cos(ang), np.sin(ang)
    t = RNG.standard_normal((1, P, 2, D))
    for pairing in ("half", "interleaved"):
        a = oracle.rope_ex(t, 1e4, pairing=pairing)
        b = oracle.rope_ex(t, 0.0, pairing=pairing, cos_tab=cos_t, sin_tab=sin_t)
        assert np.max(np.abs(a - b)) < 1e-12
        back = oracle.rope_ex(b, 0.0, sign=-1, pairing=pairing, cos_tab=cos_t, sin_tab=sin_t)
        assert np.max(np.abs(back - t)) < 1e-13
    # a table that is not a rotation (scaled cos) is applied as given
    s = oracle.rope_ex(np.ones((1, 1, 1, 2)), 0.0, cos_tab=np.array([[0.5]]), sin_tab=np.array([[0.0]]))
    assert np.allclose(s[0, 0, 0], [0.5, 0.5])


# ------------------------------------------------------- FusedLinearSwiGLU
def test_linear_swiglu_identity_weights_golden():
    g = golden("silu_values.json")
    X = np.array([[1.0, -1.0, 0.0]]); E = np.eye(3)
    out = oracle.linear_swiglu_fwd(X, E, E)                 # silu(x) * x
    assert abs(out[0, 0] - g["silu_1"]) < 1e-15 and abs(out[0, 1] - (-g["silu_m1"])) < 1e-15 and out[0, 2] == 0.0
    assert np.all(oracle.linear_swiglu_fwd(X, E, np.zeros((3, 3))) == 0.0)   # up = 0


def test_linear_swiglu_asymmetric_weights_golden():
    """Wg = I, Wu = 2I: out = silu(x) * 2x.  Swapping the gate and up roles would give
    silu(2x) * x instead (silu(2) = 1.7616 at x = 1, against 2 silu(1) = 1.4621)."""
    g = golden("silu_values.json")
    X = np.array([[1.0, -1.0, 0.0]]); E = np.eye(3)
    out = oracle.linear_swiglu_fwd(X, E, 2.0 * E)
    assert abs(out[0, 0] - 2.0 * g["silu_1"]) < 1e-15
    assert abs(out[0, 1] - (-2.0 * g["silu_m1"])) < 1e-15
    assert out[0, 2] == 0.0
    # the gate enters only through silu: gate weights 0 give silu(0) * up = 0 whatever up is,
    # while up weights 0 with a nonzero gate also give 0; a gate of 0 and up = x must give 0,
    # and a gate of x with up = 1 (a constant column) must give silu(x)
    Xc = np.array([[1.0, 1.0]])                          # column 1 is the constant 1
    Wg = np.array([[1.0, 0.0]]); Wu = np.array([[0.0, 1.0]])
    assert abs(oracle.linear_swiglu_fwd(Xc, Wg, Wu)[0, 0] - g["silu_1"]) < 1e-15
    assert abs(oracle.linear_swiglu_fwd(Xc, Wu, Wg)[0, 0] - g["silu_1"]) < 1e-15   # silu(1) * 1 both ways here
    Xd = np.array([[-1.0, 1.0]])
    assert abs(oracle.linear_swiglu_fwd(Xd, Wg, Wu)[0, 0] - g["silu_m1"]) < 1e-15   # silu(-1) * 1
    assert abs(oracle.linear_swiglu_fwd(Xd, Wu, Wg)[0, 0] - (-g["silu_1"])) < 1e-15  # silu(1) * (-1)


def _mlp_case(T=4, H=6, I=5):
    X = RNG.standard_normal((T, H)); Wg = RNG.standard_normal((I, H)); Wu = RNG.standard_normal((I, H))
    dH = RNG.standard_normal((T, I))
    return X, Wg, Wu, dH


def test_linear_swiglu_is_the_composition_of_the_pinned_steps():
    """Forward = the pinned SwiGLU applied to two library matmuls (gate X Wg^T, up X Wu^T);
    backward = the pinned SwiGLU backward pushed through the same matmuls by the chain rule."""
    X, Wg, Wu, dH = _mlp_case()
    G, U = np.matmul(X, Wg.T), np.matmul(X, Wu.T)
    assert np.max(np.abs(oracle.linear_swiglu_fwd(X, Wg, Wu) - oracle.swiglu_fwd(G, U))) < 1e-12
    dG, dU = oracle.swiglu_bwd(dH, G, U)
    dX, dWg, dWu = oracle.linear_swiglu_bwd(X, Wg, Wu, dH)
    assert np.max(np.abs(dX - (np.matmul(dG, Wg) + np.matmul(dU, Wu)))) < 1e-12
    assert np.max(np.abs(dWg - np.matmul(dG.T, X))) < 1e-12
    assert np.max(np.abs(dWu - np.matmul(dU.T, X))) < 1e-12


def test_linear_swiglu_bwd_finite_differences_of_the_composition():
    """Gradients against central differences of silu(X Wg^T) * (X Wu^T) written with numpy
    alone (sigmoid by np.exp), not the oracle's own forward."""
    X, Wg, Wu, dH = _mlp_case(3, 4, 5)
    dX, dWg, dWu = oracle.linear_swiglu_bwd(X, Wg, Wu, dH)

    def L(xx, gg, uu):
        z = np.matmul(xx, gg.T)
        return float(np.sum(dH * (z / (1.0 + np.exp(-z))) * np.matmul(xx, uu.T)))
    assert np.max(np.abs(dX - _fd(lambda v: L(v, Wg, Wu), X))) < 1e-7
    assert np.max(np.abs(dWg - _fd(lambda v: L(X, v, Wu), Wg))) < 1e-7
    assert np.max(np.abs(dWu - _fd(lambda v: L(X, Wg, v), Wu))) < 1e-7


def test_linear_swiglu_bwd_finite_differences():
    T, H, I = 3, 4, 5
    X = RNG.standard_normal((T, H)); Wg = RNG.standard_normal((I, H)); Wu = RNG.standard_normal((I, H))
    dH = RNG.standard_normal((T, I))
    dX, dWg, dWu = oracle.linear_swiglu_bwd(X, Wg, Wu, dH)
    L = lambda xx, gg, uu: float(np.sum(dH * oracle.linear_swiglu_fwd(xx, gg, uu)))
    assert np.max(np.abs(dX - _fd(lambda v: L(v, Wg, Wu), X))) < 1e-7
    assert np.max(np.abs(dWg - _fd(lambda v: L(X, v, Wu), Wg))) < 1e-7
    assert np.max(np.abs(dWu - _fd(lambda v: L(X, Wg, v), Wu))) < 1e-7


# ------------------------------------------------ fused RMSNorm + QKV + RoPE
def test_rmsnorm_qkv_rope_worked_example():
    g = golden("rmsnorm_qkv_rope_worked.json")
    A = lambda k: np.array(g[k], dtype=np.float64)
    q, k, v, rstd = oracle.rmsnorm_qkv_rope(A("x"), A("w"), A("Wq"), A("Wk"), A("Wv"), 1, 2, 1, 1, 0.0,
                                            theta=1e4, bq=A("bq"))
    assert np.allclose(rstd, 1.0, rtol=0, atol=1e-15)
    assert np.allclose(q[0, 0, 0], g["q_pos0"], atol=1e-14) and np.allclose(k[0, 0, 0], g["k_pos0"], atol=1e-14)
    assert np.allclose(q[0, 1, 0], g["q_pos1"], atol=1e-14) and np.allclose(k[0, 1, 0], g["k_pos1"], atol=1e-14)
    assert np.allclose(v[0, 0, 0], g["v"], atol=1e-14) and np.allclose(v[0, 1, 0], g["v"], atol=1e-14)


def _qkv_case(B=2, S=5, H=24, Hq=4, Hk=2, D=8, bias=True):
    x = RNG.standard_normal((B * S, H)); w = 1 + 0.1 * RNG.standard_normal(H)
    Wq = RNG.standard_normal((Hq * D, H)); Wk = RNG.standard_normal((Hk * D, H)); Wv = RNG.standard_normal((Hk * D, H))
    b = [RNG.standard_normal(n) if bias else None for n in (Hq * D, Hk * D, Hk * D)]
    return x, w, Wq, Wk, Wv, b


def test_rmsnorm_qkv_rope_is_the_composition_of_the_pinned_steps():
    """Equals RMSNorm (pinned above), a library matmul plus bias, and RoPE (pinned above)
    on q and k, with explicit positions and grouped k/v heads."""
    B, S, Hq, Hk, D, eps, theta = 2, 5, 4, 2, 8, 1e-5, 500.0
    x, w, Wq, Wk, Wv, (bq, bk, bv) = _qkv_case(B, S, 24, Hq, Hk, D)
    pos = RNG.integers(0, 4096, size=(B, S)).astype(np.int32)
    q, k, v, rstd = oracle.rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, eps, theta, bq, bk, bv, pos=pos)
    xn, r = oracle.rmsnorm_fwd(x, w, eps)
    assert np.allclose(rstd, r, rtol=1e-15)
    ql = (np.matmul(xn, Wq.T) + bq).reshape(B, S, Hq, D)
    kl = (np.matmul(xn, Wk.T) + bk).reshape(B, S, Hk, D)
    vl = (np.matmul(xn, Wv.T) + bv).reshape(B, S, Hk, D)
    assert np.max(np.abs(q - oracle.rope(ql, theta, 1, pos))) < 1e-12
    assert np.max(np.abs(k - oracle.rope(kl, theta, 1, pos))) < 1e-12
    assert np.max(np.abs(v - vl)) < 1e-12


def test_rmsnorm_qkv_rope_scale_invariance_and_relative_positions():
    B, S, Hq, Hk, D = 1, 6, 2, 1, 16
    x, w, Wq, Wk, Wv, _ = _qkv_case(B, S, 32, Hq, Hk, D, bias=False)
    q0, k0, v0, r0 = oracle.rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, 0.0, 1e4)
    q1, k1, v1, r1 = oracle.rmsnorm_qkv_rope(7.5 * x, w, Wq, Wk, Wv, B, S, Hq, Hk, 0.0, 1e4)
    assert np.max(np.abs(q1 - q0)) < 1e-12 and np.max(np.abs(v1 - v0)) < 1e-12
    assert np.allclose(r1 * 7.5, r0, rtol=1e-14)
    # every token the same row: <q_m, k_n> depends only on m - n (shift all positions by 1000)
    xs = np.repeat(x[:1], S, axis=0)
    qa, ka, _, _ = oracle.rmsnorm_qkv_rope(xs, w, Wq, Wk, Wv, B, S, Hq, Hk, 1e-6, 1e4)
    pos = (np.arange(S) + 1000).astype(np.int32).reshape(1, S)
    qb, kb, _, _ = oracle.rmsnorm_qkv_rope(xs, w, Wq, Wk, Wv, B, S, Hq, Hk, 1e-6, 1e4, pos=pos)
    da = np.einsum("mhd,nd->mnh", qa[0], ka[0, :, 0]); db = np.einsum("mhd,nd->mnh", qb[0], kb[0, :, 0])
    assert np.max(np.abs(da - db)) < 1e-9
    assert abs(da[3, 1, 0] - da[4, 2, 0]) < 1e-9 and abs(da[3, 1, 0] - da[1, 3, 0]) > 1e-6


def test_rmsnorm_qkv_rope_tables_from_the_schedule_equal_theta():
    B, S, Hq, Hk, D, theta = 1, 4, 1, 1, 8, 1e4
    x, w, Wq, Wk, Wv, (bq, bk, bv) = _qkv_case(B, S, 16, Hq, Hk, D)
    p = np.arange(16, dtype=np.float64)[:, None]; i = np.arange(D // 2, dtype=np.float64)[None, :]
    ang = p * theta ** (-2 * i / D)
    pos = np.array([[3, 0, 15, 7]], np.int32)
    b = oracle.rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, 1e-6, theta, bq, bk, bv, pos=pos,
                                cos_tab=np.cos(ang), sin_tab=np.sin(ang))
    c = oracle.rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, 1e-6, theta, bq, bk, bv, pos=pos)
    for u, z in zip(b, c):
        assert np.max(np.abs(u - z)) < 1e-12
