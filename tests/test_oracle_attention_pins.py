"""Pins for the attention oracle (``oracle.attention``): closed forms and the
finite-difference derivative, none of which retypes the oracle's formulas.

* the backward equals central finite differences of sum(o * do) in fp64, for
  q, k and v, causal and not: a dropped term, a wrong sign, a missing scale or
  a transposed operand anywhere in the backward fails it;
* causal row 0 sees only key 0: o = v[0], lse = s[0, 0];
* identical keys give uniform weights over the visible keys: o[i] is the mean
  of v[0..i], lse[i] = s + log(i + 1), and dq = 0 (the softmax gradient's rows
  sum to zero);
* one overwhelming score per row selects that row's value vector;
* lse and the probabilities agree with scipy's logsumexp / softmax on the
  masked scores;
* a planted mistake (the causal mask dropped) fails the row-0 closed form.
"""
import numpy as np
import pytest

from oracle import attention as A


def rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def loss(q, k, v, do, B, L, H, causal):
    o, _ = A.attention_forward(q, k, v, B, L, H, causal)
    return float(np.sum(o * do))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,L,H,dh", [(1, 5, 2, 4), (2, 3, 1, 6)])
def test_backward_matches_finite_differences(causal, B, L, H, dh):
    q, k, v, do = (rand((B * L, H * dh), s) for s in range(4))
    dq, dk, dv = A.attention_backward(q, k, v, do, B, L, H, causal)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            up = loss(q, k, v, do, B, L, H, causal)
            x[idx] = old - h
            dn = loss(q, k, v, do, B, L, H, causal)
            x[idx] = old
            num[idx] = (up - dn) / (2 * h)
        assert np.max(np.abs(num - g)) <= 1e-7 * max(1.0, np.max(np.abs(g)))


def test_causal_row0_sees_only_key0():
    B, L, H, dh = 2, 7, 3, 8
    q, k, v = (rand((B * L, H * dh), s) for s in range(3))
    o, lse = A.attention_forward(q, k, v, B, L, H, True)
    for b in range(B):
        row = b * L
        assert np.array_equal(o[row], v[row])
        for h in range(H):
            sl = slice(h * dh, (h + 1) * dh)
            s00 = float(np.dot(q[row, sl], k[row, sl])) / np.sqrt(dh)
            assert abs(lse[b, h, 0] - s00) <= 1e-12 * max(1.0, abs(s00))


def test_identical_keys_average_visible_values():
    B, L, H, dh = 1, 6, 2, 4
    q, v, do = (rand((B * L, H * dh), s) for s in range(3))
    k = np.tile(rand((1, H * dh), 9), (B * L, 1))
    o, lse = A.attention_forward(q, k, v, B, L, H, True)
    for i in range(L):
        assert np.allclose(o[i], v[: i + 1].mean(axis=0), rtol=0, atol=1e-12)
        for h in range(H):
            sl = slice(h * dh, (h + 1) * dh)
            s = float(np.dot(q[i, sl], k[0, sl])) / np.sqrt(dh)
            assert abs(lse[0, h, i] - (s + np.log(i + 1))) <= 1e-12
    dq, _, _ = A.attention_backward(q, k, v, do, B, L, H, True)
    assert np.max(np.abs(dq)) <= 1e-12


def test_overwhelming_score_selects_value():
    B, L, H, dh = 1, 6, 1, 8
    k = np.zeros((L, dh))
    k[np.arange(L), np.arange(L)] = 10.0          # key j points along axis j
    target = [0, 0, 1, 3, 2, 5]                   # a visible key for every row
    q = np.zeros((L, dh))
    q[np.arange(L), target] = 100.0               # score 1000 / sqrt(8) on the target
    v = rand((L, dh), 3)
    o, _ = A.attention_forward(q, k, v, B, L, H, True)
    assert np.allclose(o, v[target], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_matches_scipy_softmax(causal):
    sp = pytest.importorskip("scipy.special")
    B, L, H, dh = 2, 9, 2, 8
    q, k = (rand((B * L, H * dh), s) for s in range(2))
    s = A.scores(q, k, B, L, H)
    p, lse = A.probabilities(s, causal)
    mask = np.tril(np.ones((L, L), bool)) if causal else np.ones((L, L), bool)
    masked = np.where(mask, s, -np.inf)
    assert np.allclose(lse, sp.logsumexp(masked, axis=-1), rtol=0, atol=1e-12)
    assert np.allclose(p, sp.softmax(masked, axis=-1), rtol=0, atol=1e-14)


def test_rowdot_is_the_softmax_gradient_row_term():
    B, L, H, dh = 2, 5, 2, 4
    q, k, v, do = (rand((B * L, H * dh), s) for s in range(4))
    o, _ = A.attention_forward(q, k, v, B, L, H, True)
    p, _ = A.probabilities(A.scores(q, k, B, L, H), True)
    vh, doh = A._heads(v, B, L, H), A._heads(do, B, L, H)
    dp = np.einsum("bhie,bhje->bhij", doh, vh)
    assert np.allclose(A.rowdot(o, do, B, L, H), (p * dp).sum(-1), rtol=0, atol=1e-12)


def test_planted_mask_mistake_fails_row0(monkeypatch):
    monkeypatch.setattr(A, "_allowed", lambda L, causal: np.ones((L, L), dtype=bool))
    B, L, H, dh = 1, 4, 1, 4
    q, k, v = (rand((B * L, H * dh), s) for s in range(3))
    o, _ = A.attention_forward(q, k, v, B, L, H, True)
    assert np.max(np.abs(o[0] - v[0])) > 1e-3
