"""Pins for the oracle with bottlenecks of uneven size (each factorised layer its
own rank r_i; BOOST page, Limitations -> "Untested extensions": the design also
covers bottlenecks of different sizes). Each check compares the oracle with
something other than itself:

* central finite differences of the loss for every parameter and the input,
  with seven different ranks (a wrong split of the grouped Q/K/V or gate/up
  tensors breaks the shapes or the derivatives);
* zero padding: giving layer i extra rank directions whose A rows and B columns
  are zero leaves every output and every gradient of the original entries
  unchanged and gives zero gradients to the padded ones -- which pins where the
  grouped tensors are split;
* checkpoint mode saves exactly sum(r_i) values per token;
* the BTP data flow with uneven ranks equals the plain block, and its r-wide
  all-reduces carry sum(r_i) values per token and pass.
"""
import numpy as np
import pytest

import oracle as O
from oracle import btp as OB
from rank_bottleneck_gb300.synth import make_block_inputs

RANKS = (2, 3, 1, 4, 2, 3, 1)  # q, k, v, o, gate, up, down


def inputs(T, d, r, d_ff, ranks, kind="full", seed=0):
    a = {k: v.astype(np.float64) for k, v in
         make_block_inputs(T, d, r, d_ff, kind=kind, dtype="f32", seed=seed, ranks=ranks).items()}
    x, dy = a.pop("x"), a.pop("dy")
    return a, x, dy, a.pop("dq", None), a.pop("dk", None)


@pytest.mark.parametrize("cfg", [dict(kind="full"), dict(kind="full", checkpoint=True),
                                 dict(kind="full", sigma="identity"), dict(kind="mlp")],
                         ids=lambda c: "-".join(f"{k}={v}" for k, v in c.items()))
def test_uneven_ranks_finite_differences(cfg):
    T, d, d_ff = 3, 8, 7
    p, x, dy, dq, dk = inputs(T, d, 2, d_ff, RANKS, kind=cfg["kind"], seed=4)
    p = {k: (v * 1.7 if k.startswith(("A_", "B_")) else v) for k, v in p.items()}
    _, saved = O.block_forward(p, x, cfg)
    dx, g = O.block_backward(p, x, saved, dy, dq, dk, cfg)
    h = 1e-6

    def fd(get, put, shape, xx):
        out = np.zeros(shape)
        for idx in np.ndindex(*shape):
            base = get()[idx]
            put(idx, base + h)
            lp = O.loss(p, xx, dy, dq, dk, cfg)
            put(idx, base - h)
            lm = O.loss(p, xx, dy, dq, dk, cfg)
            put(idx, base)
            out[idx] = (lp - lm) / (2 * h)
        return out

    xv = x.copy()
    fdx = fd(lambda: xv, lambda i, v: xv.__setitem__(i, v), x.shape, xv)
    assert np.max(np.abs(dx - fdx)) <= 1e-6 * max(1.0, np.max(np.abs(fdx)))
    assert set(g) == set(p)
    for name in g:
        assert g[name].shape == p[name].shape, name
        fdp = fd(lambda n=name: p[n], lambda i, v, n=name: p[n].__setitem__(i, v), p[name].shape, x)
        err = np.max(np.abs(g[name] - fdp))
        assert err <= 1e-6 * max(1.0, np.max(np.abs(fdp))), (name, err)


def _pad(p, r, extra):
    """The rank-r parameters with layer i widened by extra[i] zero directions
    (zero A rows, zero B columns), grouped tensors kept in layer order."""
    rq, rk, rv, ro, rg, ru, rd = [r + e for e in extra]
    q = dict(p)

    def grow_rows(A, n):
        return np.concatenate([A, np.zeros((n, A.shape[1]))], axis=0)

    def grow_cols(B, n):
        return np.concatenate([B, np.zeros((B.shape[0], n))], axis=1)

    if "A_qkv" in p:
        Aq, Ak, Av = np.split(p["A_qkv"], 3, axis=0)
        q["A_qkv"] = np.concatenate([grow_rows(Aq, extra[0]), grow_rows(Ak, extra[1]),
                                     grow_rows(Av, extra[2])], axis=0)
        q["B_q"], q["B_k"], q["B_v"] = (grow_cols(p["B_q"], extra[0]), grow_cols(p["B_k"], extra[1]),
                                        grow_cols(p["B_v"], extra[2]))
        q["A_o"], q["B_o"] = grow_rows(p["A_o"], extra[3]), grow_cols(p["B_o"], extra[3])
    Ag, Au = np.split(p["A_gu"], 2, axis=0)
    q["A_gu"] = np.concatenate([grow_rows(Ag, extra[4]), grow_rows(Au, extra[5])], axis=0)
    q["B_g"], q["B_u"] = grow_cols(p["B_g"], extra[4]), grow_cols(p["B_u"], extra[5])
    q["A_d"], q["B_d"] = grow_rows(p["A_d"], extra[6]), grow_cols(p["B_d"], extra[6])
    assert q["B_q" if "B_q" in q else "B_g"].shape[1] == (rq if "B_q" in q else rg)
    return q


@pytest.mark.parametrize("kind", ["full", "mlp"])
@pytest.mark.parametrize("sigma", ["silu", "identity"])
def test_zero_padded_ranks_reduce_to_the_even_block(kind, sigma):
    T, d, r, d_ff = 10, 16, 4, 24
    extra = (8, 0, 4, 12, 4, 8, 16)
    p, x, dy, dq, dk = inputs(T, d, r, d_ff, None, kind=kind, seed=9)
    q = _pad(p, r, extra)
    cfg = dict(kind=kind, sigma=sigma)
    out_p, sv_p = O.block_forward(p, x, cfg)
    out_q, sv_q = O.block_forward(q, x, cfg)
    for k in out_p:
        np.testing.assert_allclose(out_q[k], out_p[k], rtol=1e-12, atol=1e-12)
    dx_p, g_p = O.block_backward(p, x, sv_p, dy, dq, dk, cfg)
    dx_q, g_q = O.block_backward(q, x, sv_q, dy, dq, dk, cfg)
    np.testing.assert_allclose(dx_q, dx_p, rtol=1e-12, atol=1e-12)
    for name, gp in g_p.items():
        gq = g_q[name]
        if name.startswith("w_"):
            np.testing.assert_allclose(gq, gp, rtol=1e-12, atol=1e-12)
            continue
        # the original entries agree; the padded ones get zero gradient
        mask = np.zeros(gq.shape, dtype=bool)
        idx = _orig_index(name, r, extra, gq.shape)
        mask[idx] = True
        np.testing.assert_allclose(gq[mask].reshape(gp.shape), gp, rtol=1e-12, atol=1e-12)
        assert np.all(gq[~mask] == 0.0), name


def _orig_index(name, r, extra, shape):
    """Index of the rank-r entries inside the padded parameter `name`."""
    layer = dict(B_q=0, B_k=1, B_v=2, A_o=3, B_o=3, B_g=4, B_u=5, A_d=6, B_d=6)
    if name in ("A_qkv", "A_gu"):
        ex = extra[0:3] if name == "A_qkv" else extra[4:6]
        rows, base = [], 0
        for e in ex:
            rows += list(range(base, base + r))
            base += r + e
        return (np.array(rows)[:, None], np.arange(shape[1])[None, :])
    if name.startswith("A_"):
        return (np.arange(r)[:, None], np.arange(shape[1])[None, :])
    return (np.arange(shape[0])[:, None], np.arange(r)[None, :])


def test_checkpoint_saves_the_sum_of_the_ranks():
    T, d, d_ff = 4, 16, 20
    ranks = (8, 16, 24, 8, 32, 16, 8)
    p, x, *_ = inputs(T, d, 8, d_ff, ranks)
    _, saved = O.block_forward(p, x, dict(checkpoint=True))
    assert sum(v.shape[1] for v in saved.values()) == sum(ranks)


@pytest.mark.parametrize("kind", ["full", "mlp"])
def test_btp_with_uneven_ranks_equals_plain_and_carries_sum_of_ranks(kind):
    T, d, d_ff, S = 6, 16, 24, 4
    ranks = (8, 16, 24, 8, 32, 16, 8)
    p, x, dy, dq, dk = inputs(T, d, 8, d_ff, ranks, kind=kind, seed=2)
    cfg = dict(kind=kind)
    out, saved = O.block_forward(p, x, cfg)
    dx, g = O.block_backward(p, x, saved, dy, dq, dk, cfg)
    out_b, acts, vol_f = OB.block_forward_btp(p, x, S, cfg)
    dx_b, g_b, vol_b = OB.block_backward_btp(p, x, acts, dy, S, dq, dk, cfg)
    for k in out:
        np.testing.assert_allclose(out_b[k], out[k], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dx_b, dx, rtol=1e-12, atol=1e-12)
    for k in g:
        np.testing.assert_allclose(g_b[k], g[k], rtol=1e-12, atol=1e-12)
    want = sum(ranks) if kind == "full" else sum(ranks[4:])
    assert vol_f["r_wide"] == want and vol_b["r_wide"] == want
