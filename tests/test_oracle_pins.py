"""Pins for the fp64 oracle: every check compares it with something other than itself.

* closed forms and special values (SiLU at 0 and +-ln 3, RMSNorm of rows with a
  known mean square),
* brute-force loops on tiny inputs,
* the exactness of Online RMSNorm (BOOST, "Three supporting changes" -> Online
  RMSNorm; BOOST-MLSys26 core method: mathematically equivalent) for every S,
* the reduction to a dense layer when r = d and sigma = identity,
* central finite differences of the loss for every parameter and the input,
* checkpoint (recompute) versus stored activations, bit for bit,
* the page's printed volume table and parameter ratio.
"""
import math
import os

import numpy as np
import pytest

import oracle as O
from rank_bottleneck_gb300.synth import make_block_inputs, round_to_bf16, tensor_shapes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(d):
    return {k: v.astype(np.float64) for k, v in d.items()}


def split_inputs(T, d, r, d_ff, kind="full", dense=False, seed=0, dtype="f32"):
    a = f64(make_block_inputs(T, d, r, d_ff, kind=kind, dense=dense, dtype=dtype, seed=seed))
    x, dy = a.pop("x"), a.pop("dy")
    dq, dk = a.pop("dq", None), a.pop("dk", None)
    return a, x, dy, dq, dk


# ---------------------------------------------------------------------------
# elementwise pieces
# ---------------------------------------------------------------------------

def test_silu_special_values():
    ln3 = math.log(3.0)  # sigmoid(ln 3) = 3/4 exactly
    assert O.silu(np.array(0.0)) == 0.0
    np.testing.assert_allclose(O.silu(np.array(ln3)), 0.75 * ln3, rtol=1e-15)
    np.testing.assert_allclose(O.silu(np.array(-ln3)), -0.25 * ln3, rtol=1e-15)
    np.testing.assert_allclose(O.silu_grad(np.array(ln3)), 0.75 * (1 + 0.25 * ln3), rtol=1e-15)
    assert O.silu_grad(np.array(0.0)) == 0.5
    assert abs(O.silu(np.array(40.0)) - 40.0) < 1e-12      # -> z for large z
    assert abs(O.silu(np.array(-40.0))) < 1e-12            # -> 0 for very negative z


def test_silu_grad_matches_finite_differences():
    z = np.linspace(-7, 7, 141)
    h = 1e-6
    fd = (O.silu(z + h) - O.silu(z - h)) / (2 * h)
    np.testing.assert_allclose(O.silu_grad(z), fd, atol=1e-9)
    assert np.all(O.act_grad(z, "identity") == 1.0)
    assert np.array_equal(O.act(z, "identity"), z)


def test_swiglu_definition_and_grad():
    rng = np.random.default_rng(1)
    G, U, dm = rng.standard_normal((3, 5, 7))
    m = O.swiglu(G, U)
    np.testing.assert_allclose(m, G / (1 + np.exp(-G)) * U, rtol=1e-14)
    dG, dU = O.swiglu_backward(dm, G, U)
    h = 1e-6
    fdG = (np.sum(O.swiglu(G + h, U) * dm, axis=None) - np.sum(O.swiglu(G - h, U) * dm)) / (2 * h)
    np.testing.assert_allclose(np.sum(dG), fdG, rtol=1e-7)
    fdU = (np.sum(O.swiglu(G, U + h) * dm) - np.sum(O.swiglu(G, U - h) * dm)) / (2 * h)
    np.testing.assert_allclose(np.sum(dU), fdU, rtol=1e-7)


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rmsnorm_closed_forms():
    w = np.array([1.0, 2.0, -0.5, 3.0])
    x = np.array([[3.0, 4.0, 0.0, 0.0]])  # mean square 25/4 -> rms 2.5
    n, rstd = O.rmsnorm(x, w, eps=0.0)
    np.testing.assert_allclose(rstd, [[0.4]], rtol=1e-15)
    np.testing.assert_allclose(n, [[1.2, 3.2, 0.0, 0.0]], rtol=1e-15)
    c = 0.01  # constant row: rms = sqrt(c^2 + eps), eps inside the square root
    n, _ = O.rmsnorm(np.full((1, 4), c), w, eps=1e-5)
    np.testing.assert_allclose(n, c * w[None] / math.sqrt(c * c + 1e-5), rtol=1e-14)


def test_rmsnorm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 32))
    w = np.ones(32)
    n1, _ = O.rmsnorm(x, w, eps=0.0)
    n2, _ = O.rmsnorm(37.5 * x, w, eps=0.0)
    np.testing.assert_allclose(n1, n2, rtol=1e-13)
    np.testing.assert_allclose(np.sqrt(np.mean(n1 * n1, axis=1)), 1.0, rtol=1e-13)


def test_rmsnorm_backward_finite_differences():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 10))
    w = 1 + 0.1 * rng.standard_normal(10)
    dn = rng.standard_normal((4, 10))
    _, rstd = O.rmsnorm(x, w)
    dx, dw = O.rmsnorm_backward(dn, x, w, rstd)
    h = 1e-6

    def L(xx, ww):
        return np.sum(O.rmsnorm(xx, ww)[0] * dn)

    fdx = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        e = np.zeros_like(x)
        e[idx] = h
        fdx[idx] = (L(x + e, w) - L(x - e, w)) / (2 * h)
    fdw = np.array([(L(x, w + h * np.eye(10)[j]) - L(x, w - h * np.eye(10)[j])) / (2 * h)
                    for j in range(10)])
    np.testing.assert_allclose(dx, fdx, atol=1e-8)
    np.testing.assert_allclose(dw, fdw, atol=1e-8)


# ---------------------------------------------------------------------------
# Online RMSNorm: exact for every S
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 2, 4, 8])
@pytest.mark.parametrize("scale", [1.0, 1e-3])
def test_online_rmsnorm_equals_plain(S, scale):
    rng = np.random.default_rng(4 + S)
    T, d, n_out = 9, 64, 24
    x = scale * rng.standard_normal((T, d))
    x[:, : d // 8] *= 50.0  # shards of very different magnitude
    x[1, : d // S] = 0.0    # a row whose first shard is all zeros (local RMS = sqrt(eps))
    x[2, :] = 0.0           # an all-zero row
    w = 1 + 0.1 * rng.standard_normal(d)
    A = rng.standard_normal((n_out, d)) / math.sqrt(d)
    ref = O.rmsnorm(x, w)[0] @ A.T
    got = O.online_rmsnorm_linear(x, w, A, S)
    assert np.all(np.isfinite(got)) and np.all(got[2] == 0.0)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_online_rmsnorm_rejects_uneven_split():
    with pytest.raises(ValueError):
        O.online_rmsnorm_linear(np.ones((2, 10)), np.ones(10), np.ones((3, 10)), 4)


# ---------------------------------------------------------------------------
# one bottleneck layer: brute force and the dense reduction
# ---------------------------------------------------------------------------

def test_lowrank_forward_brute_force():
    rng = np.random.default_rng(5)
    T, d_in, r, d_out = 3, 4, 2, 5
    X = rng.standard_normal((T, d_in))
    A = rng.standard_normal((r, d_in))
    B = rng.standard_normal((d_out, r))
    out, z, h = O.lowrank_forward(X, A, B, "silu")
    for t in range(T):
        for j in range(r):
            zz = sum(A[j, i] * X[t, i] for i in range(d_in))
            assert abs(z[t, j] - zz) < 1e-13
            assert abs(h[t, j] - zz / (1 + math.exp(-zz))) < 1e-13
        for o in range(d_out):
            acc = sum(B[o, j] * (z[t, j] / (1 + math.exp(-z[t, j]))) for j in range(r))
            assert abs(out[t, o] - acc) < 1e-12


def _dense_from_lowrank(p, r):
    """W = B . A per layer (sigma = identity, r = d): the full-rank equivalent block."""
    A_q, A_k, A_v = np.split(p["A_qkv"], 3, axis=0)
    A_g, A_u = np.split(p["A_gu"], 2, axis=0)
    return dict(w_norm1=p["w_norm1"], w_norm2=p["w_norm2"],
                A_qkv=np.concatenate([p["B_q"] @ A_q, p["B_k"] @ A_k, p["B_v"] @ A_v]),
                A_o=p["B_o"] @ p["A_o"],
                A_gu=np.concatenate([p["B_g"] @ A_g, p["B_u"] @ A_u]),
                A_d=p["B_d"] @ p["A_d"])


def test_full_rank_reduction_block():
    T, d, d_ff = 7, 16, 24
    r = d
    p, x, dy, dq, dk = split_inputs(T, d, r, d_ff)
    # the MLP down factor is [r, d_ff] with r = d here
    cfg_lr = dict(sigma="identity")
    out_lr, saved_lr = O.block_forward(p, x, cfg_lr)
    pd = _dense_from_lowrank(p, r)
    out_dn, saved_dn = O.block_forward(pd, x, dict(dense=True))
    for k in out_lr:
        np.testing.assert_allclose(out_lr[k], out_dn[k], rtol=1e-11, atol=1e-11)
    dx_lr, g_lr = O.block_backward(p, x, saved_lr, dy, dq, dk, cfg_lr)
    dx_dn, g_dn = O.block_backward(pd, x, saved_dn, dy, dq, dk, dict(dense=True))
    np.testing.assert_allclose(dx_lr, dx_dn, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(g_lr["w_norm1"], g_dn["w_norm1"], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(g_lr["w_norm2"], g_dn["w_norm2"], rtol=1e-10, atol=1e-10)
    # dA = B^T dW and dB = dW A^T for each factor pair
    dWo = g_dn["A_o"]
    np.testing.assert_allclose(g_lr["A_o"], p["B_o"].T @ dWo, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(g_lr["B_o"], dWo @ p["A_o"].T, rtol=1e-10, atol=1e-10)
    dWd = g_dn["A_d"]
    np.testing.assert_allclose(g_lr["A_d"], p["B_d"].T @ dWd, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(g_lr["B_d"], dWd @ p["A_d"].T, rtol=1e-10, atol=1e-10)
    dWq = np.split(g_dn["A_qkv"], 3, axis=0)[0]
    A_q = np.split(p["A_qkv"], 3, axis=0)[0]
    np.testing.assert_allclose(np.split(g_lr["A_qkv"], 3, axis=0)[0], p["B_q"].T @ dWq,
                               rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(g_lr["B_q"], dWq @ A_q.T, rtol=1e-10, atol=1e-10)
    dWu = np.split(g_dn["A_gu"], 2, axis=0)[1]
    A_u = np.split(p["A_gu"], 2, axis=0)[1]
    np.testing.assert_allclose(g_lr["B_u"], dWu @ A_u.T, rtol=1e-10, atol=1e-10)


def _silu(v):
    return v / (1 + math.exp(-v))


@pytest.mark.parametrize("ranks", [None, (2, 1, 3, 2, 1, 3, 2)])
def test_full_block_forward_brute_force(ranks):
    """The whole factorised block (attention core outside: O reads V), every
    token row and every output element of y, q, k written out as loops over the
    definition: RMSNorm, the grouped Q/K/V bottlenecks, O, the residual, RMSNorm,
    gate/up, SwiGLU, down, the residual -- with equal and with uneven ranks."""
    T, d, r, d_ff = 3, 4, 2, 5
    a = f64(make_block_inputs(T, d, r, d_ff, dtype="f32", seed=13, ranks=ranks))
    p = {k: v for k, v in a.items() if k not in ("x", "dy", "dq", "dk")}
    x = a["x"]
    out, _ = O.block_forward(p, x, dict(kind="full"))
    rq, rk, rv = p["B_q"].shape[1], p["B_k"].shape[1], p["B_v"].shape[1]
    ro, rg, ru, rd = p["A_o"].shape[0], p["B_g"].shape[1], p["B_u"].shape[1], p["A_d"].shape[0]

    def norm(row, w):
        ms = sum(v * v for v in row) / len(row)
        return [row[j] * w[j] / math.sqrt(ms + O.EPS) for j in range(len(row))]

    def lin(W, v):  # W [out, in] times the vector v
        return [sum(W[o][i] * v[i] for i in range(len(v))) for o in range(len(W))]

    for t in range(T):
        n1 = norm(list(x[t]), p["w_norm1"])
        h = [_silu(z) for z in lin(p["A_qkv"], n1)]
        q = lin(p["B_q"], h[:rq])
        k = lin(p["B_k"], h[rq:rq + rk])
        v = lin(p["B_v"], h[rq + rk:rq + rk + rv])
        ho = [_silu(z) for z in lin(p["A_o"], v)]
        x1 = [x[t][o] + sum(p["B_o"][o][c] * ho[c] for c in range(ro)) for o in range(d)]
        n2 = norm(x1, p["w_norm2"])
        hgu = [_silu(z) for z in lin(p["A_gu"], n2)]
        G = lin(p["B_g"], hgu[:rg])
        U = lin(p["B_u"], hgu[rg:rg + ru])
        m = [_silu(G[i]) * U[i] for i in range(d_ff)]
        hd = [_silu(z) for z in lin(p["A_d"], m)]
        y = [x1[o] + sum(p["B_d"][o][c] * hd[c] for c in range(rd)) for o in range(d)]
        np.testing.assert_allclose(out["q"][t], q, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out["k"][t], k, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out["y"][t], y, rtol=1e-12, atol=1e-14)


def test_dense_layer_brute_force():
    # the dense path the reduction compares against: y = x1 + m W_d^T, one entry by loops
    T, d, d_ff = 2, 4, 6
    p, x, dy, dq, dk = split_inputs(T, d, 4, d_ff, kind="mlp", dense=True)
    out, a = O.block_forward(p, x, dict(kind="mlp", dense=True))
    ms = [sum(x[0, j] ** 2 for j in range(d)) / d]
    n = [x[0, j] * p["w_norm2"][j] / math.sqrt(ms[0] + O.EPS) for j in range(d)]
    gu = [sum(p["A_gu"][o, j] * n[j] for j in range(d)) for o in range(2 * d_ff)]
    m = [gu[i] / (1 + math.exp(-gu[i])) * gu[d_ff + i] for i in range(d_ff)]
    y0 = [x[0, o] + sum(p["A_d"][o, i] * m[i] for i in range(d_ff)) for o in range(d)]
    np.testing.assert_allclose(out["y"][0], y0, rtol=1e-12)


# ---------------------------------------------------------------------------
# finite differences of the whole block
# ---------------------------------------------------------------------------

FD_CASES = [
    dict(kind="full", sigma="silu"),
    dict(kind="full", sigma="identity"),
    dict(kind="full", sigma="silu", checkpoint=True),
    dict(kind="mlp", sigma="silu"),
    dict(kind="mlp", sigma="silu", checkpoint=True),
    dict(kind="full", dense=True),
    dict(kind="mlp", dense=True),
    # the causal attention core inside the block: one sequence of the 3 tokens,
    # 2 heads of 4
    dict(kind="full", sigma="silu", attn=True, seq_len=3, heads=2),
    dict(kind="full", sigma="silu", attn=True, seq_len=3, heads=2, checkpoint=True),
    dict(kind="full", dense=True, attn=True, seq_len=3, heads=2),
]


@pytest.mark.parametrize("cfg", FD_CASES, ids=lambda c: "-".join(f"{k}={v}" for k, v in c.items()))
@pytest.mark.parametrize("d_ff", [12, 7])
def test_block_gradients_finite_differences(cfg, d_ff):
    T, d, r = 3, 8, 2
    p, x, dy, dq, dk = split_inputs(T, d, r, d_ff, kind=cfg["kind"],
                                    dense=cfg.get("dense", False), seed=11)
    # larger-than-init weights so every nonlinearity is exercised away from 0
    p = {k: (v * 1.7 if k.startswith(("A_", "B_")) else v) for k, v in p.items()}
    _, saved = O.block_forward(p, x, cfg)
    dx, g = O.block_backward(p, x, saved, dy, dq, dk, cfg)
    h = 1e-6

    def fd(arr_get, arr_set, shape):
        out = np.zeros(shape)
        for idx in np.ndindex(*shape):
            base = arr_get()[idx]
            arr_set(idx, base + h)
            lp = O.loss(p, xv[0], dy, dq, dk, cfg)
            arr_set(idx, base - h)
            lm = O.loss(p, xv[0], dy, dq, dk, cfg)
            arr_set(idx, base)
            out[idx] = (lp - lm) / (2 * h)
        return out

    xv = [x.copy()]

    def setx(idx, v):
        xv[0][idx] = v
    fdx = fd(lambda: xv[0], setx, x.shape)
    assert np.max(np.abs(dx - fdx)) <= 1e-6 * max(1.0, np.max(np.abs(fdx)))
    for name in g:
        def setp(idx, v, name=name):
            p[name][idx] = v
        fdp = fd(lambda name=name: p[name], setp, p[name].shape)
        err = np.max(np.abs(g[name] - fdp))
        assert err <= 1e-6 * max(1.0, np.max(np.abs(fdp))), (name, err)
    # every parameter has a gradient
    assert set(g) == set(p)


# ---------------------------------------------------------------------------
# checkpointing: recomputed == stored, bit for bit
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["full", "mlp"])
def test_checkpoint_recompute_is_bit_identical(kind):
    T, d, r, d_ff = 16, 32, 8, 40
    p, x, dy, dq, dk = split_inputs(T, d, r, d_ff, kind=kind, seed=3)
    out_a, saved_a = O.block_forward(p, x, dict(kind=kind))
    out_b, saved_b = O.block_forward(p, x, dict(kind=kind, checkpoint=True))
    assert set(saved_b) == ({"z_qkv", "z_o", "z_gu", "z_d"} if kind == "full" else {"z_gu", "z_d"})
    for k in out_a:
        assert np.array_equal(out_a[k], out_b[k])
    dx_a, g_a = O.block_backward(p, x, saved_a, dy, dq, dk, dict(kind=kind))
    dx_b, g_b = O.block_backward(p, x, saved_b, dy, dq, dk, dict(kind=kind, checkpoint=True))
    assert np.array_equal(dx_a, dx_b)
    for k in g_a:
        assert np.array_equal(g_a[k], g_b[k]), k
    # the recomputed activations equal the stored ones
    rec = O.recompute(p, x, saved_b, dict(kind=kind, checkpoint=True))
    for k in ("x1", "m", "G", "U", "h_d", "h_gu"):
        assert np.array_equal(rec[k], saved_a[k]), k


def test_checkpoint_saved_width_is_7r():
    T, d, r, d_ff = 4, 16, 4, 20
    p, x, *_ = split_inputs(T, d, r, d_ff)
    _, saved = O.block_forward(p, x, dict(checkpoint=True))
    assert sum(v.shape[1] for v in saved.values()) == 7 * r
    assert all(v.shape[0] == T for v in saved.values())


# ---------------------------------------------------------------------------
# the page's printed volume table and parameter ratio
# ---------------------------------------------------------------------------

def _golden_table():
    vals = {}
    with open(os.path.join(GOLDEN, "volume_table.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            vals[parts[0]] = parts[1:]
    return vals


def test_volume_table_and_param_ratio_from_layer_set():
    g = _golden_table()
    d, d_ff, r = int(g["d"][0]), int(g["d_ff"][0]), int(g["r"][0])
    shapes = {n: s for n, s, _ in tensor_shapes(1, d, r, d_ff)}
    # BOOST all-reduces once per chunk, at the r-wide output of each down-projection
    down_widths = sum(shapes[n][0] for n in ("A_qkv", "A_o", "A_gu", "A_d"))
    # vanilla low-rank TP all-reduces the full-width output of each up-projection
    up_widths = sum(shapes[n][0] for n in ("B_q", "B_k", "B_v", "B_o", "B_g", "B_u", "B_d"))
    assert down_widths == 7 * r and up_widths == 5 * d + 2 * d_ff
    full = 2 * d
    assert round(up_widths / full, 2) == float(g["vanilla_lowrank"][1])
    assert round(down_widths / full, 2) == float(g["boost"][1])
    # parameter count: dense block versus factorised block
    dense = {n: s for n, s, _ in tensor_shapes(1, d, r, d_ff, dense=True)}
    n_dense = sum(np.prod(dense[n]) for n in ("A_qkv", "A_o", "A_gu", "A_d"))
    n_lr = sum(np.prod(shapes[n]) for n in shapes if n.startswith(("A_", "B_")))
    assert abs(n_dense / n_lr - float(g["param_ratio_about"][0])) < 0.05


# ---------------------------------------------------------------------------
# the shared input generator
# ---------------------------------------------------------------------------

def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    v = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    v[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]  # exact ties round to even
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(round_to_bf16(v), ref)


def test_generator_is_deterministic_and_ordered():
    a = make_block_inputs(8, 16, 4, 24, seed=5)
    b = make_block_inputs(8, 16, 4, 24, seed=5)
    assert list(a) == ["x", "w_norm1", "A_qkv", "B_q", "B_k", "B_v", "A_o", "B_o", "w_norm2",
                       "A_gu", "B_g", "B_u", "A_d", "B_d", "dy", "dq", "dk"]
    for k in a:
        assert np.array_equal(a[k], b[k])
        assert np.array_equal(round_to_bf16(a[k]), a[k])  # bf16 by default
    m = make_block_inputs(8, 16, 4, 24, kind="mlp", seed=5)
    assert np.array_equal(m["x"], a["x"])
    assert "dq" not in m and "A_qkv" not in m


def test_attention_inside_block_two_sequences_do_not_mix():
    """With the attention core inside, a token's output depends on its own
    sequence only (causal within each of the T / seq_len sequences): changing
    the second sequence leaves the first one's outputs as they were, and
    changing a later token leaves earlier tokens of its sequence unchanged."""
    T, d, r, d_ff = 8, 16, 4, 12
    cfg = dict(kind="full", attn=True, seq_len=4, heads=2)
    p, x, dy, dq, dk = split_inputs(T, d, r, d_ff, kind="full", seed=5)
    y0 = O.block_forward(p, x, cfg)[0]["y"]
    x2 = x.copy()
    x2[6] += 1.0                      # the second sequence's third token
    y1 = O.block_forward(p, x2, cfg)[0]["y"]
    assert np.array_equal(y0[:6], y1[:6])
    assert np.max(np.abs(y0[6:] - y1[6:])) > 1e-3
