"""fp64 CPU oracle for the attention core that sits between the block's grouped
Q/K/V up-projection and its O projection.

TEST INFRASTRUCTURE ONLY. Imported by ``tests/`` and by the CPU legs of
``bench.py``; the library never imports or calls it, and it imports nothing
from the library.

What it computes. The pages name the attention core only as the step between
the Q/K/V projections and the O projection of the LLaMA decoder block (BOOST,
"Move the chunk boundary to the bottleneck", the decoder-block figure) and
cite FlashAttention for it (BOOST-MLSys26, references); they give no formula.
The plainest reading is exact multi-head causal softmax attention, which is
what FlashAttention computes:

    s[b, h, i, j] = scale * sum_e q[b, i, h, e] * k[b, j, h, e],  scale = 1 / sqrt(d_head)
    allowed(i, j) = j <= i (causal) or always (non-causal)
    lse[b, h, i]  = log sum_{allowed j} exp(s[b, h, i, j])
    p[b, h, i, j] = exp(s[b, h, i, j] - lse[b, h, i]) on allowed (i, j), else 0
    o[b, i, h, :] = sum_j p[b, h, i, j] * v[b, j, h, :]

The backward is the plain derivative of that definition for an upstream
gradient do:

    dv[j] = sum_i p[i, j] do[i]
    dp[i, j] = do[i] . v[j]
    ds[i, j] = p[i, j] (dp[i, j] - sum_j' p[i, j'] dp[i, j'])
    dq[i] = scale sum_j ds[i, j] k[j],   dk[j] = scale sum_i ds[i, j] q[i]

Layout: q, k, v, o, do and the gradients are [T, H * d_head] with T = B * L
token rows (sequence b occupies rows b L .. b L + L - 1; head h columns
h d_head .. h d_head + d_head - 1), the layout the block's Q/K/V up-projection
writes. lse is [B, H, L]. Precision: float64 throughout; bf16 inputs arrive
already rounded and are never rounded again.
"""
from __future__ import annotations

import numpy as np


def _heads(x, B, L, H):
    """[T, H * dh] -> [B, H, L, dh] (a view reshaped; no arithmetic)."""
    T, D = x.shape
    assert T == B * L and D % H == 0
    return np.asarray(x, dtype=np.float64).reshape(B, L, H, D // H).transpose(0, 2, 1, 3)


def _tokens(x):
    """[B, H, L, dh] -> [T, H * dh]."""
    B, H, L, dh = x.shape
    return np.ascontiguousarray(x.transpose(0, 2, 1, 3)).reshape(B * L, H * dh)


def _allowed(L, causal):
    if causal:
        return np.tril(np.ones((L, L), dtype=bool))
    return np.ones((L, L), dtype=bool)


def scores(q, k, B, L, H):
    """s [B, H, L, L] = scale q k^T per head, scale = 1 / sqrt(d_head)."""
    qh, kh = _heads(q, B, L, H), _heads(k, B, L, H)
    scale = 1.0 / np.sqrt(qh.shape[-1])
    return scale * np.einsum("bhie,bhje->bhij", qh, kh)


def probabilities(s, causal):
    """Row softmax over the allowed keys; returns (p, lse)."""
    L = s.shape[-1]
    mask = _allowed(L, causal)
    masked = np.where(mask, s, -np.inf)
    mx = masked.max(axis=-1, keepdims=True)
    e = np.where(mask, np.exp(masked - mx), 0.0)
    tot = e.sum(axis=-1, keepdims=True)
    lse = (mx + np.log(tot))[..., 0]
    return e / tot, lse


def attention_forward(q, k, v, B, L, H, causal=True):
    """Returns (o [T, H dh], lse [B, H, L])."""
    p, lse = probabilities(scores(q, k, B, L, H), causal)
    o = np.einsum("bhij,bhje->bhie", p, _heads(v, B, L, H))
    return _tokens(o), lse


def attention_backward(q, k, v, do, B, L, H, causal=True):
    """Returns (dq, dk, dv), each [T, H dh], for the upstream gradient do."""
    qh, kh, vh, doh = (_heads(x, B, L, H) for x in (q, k, v, do))
    scale = 1.0 / np.sqrt(qh.shape[-1])
    p, _ = probabilities(scores(q, k, B, L, H), causal)
    dv = np.einsum("bhij,bhie->bhje", p, doh)
    dp = np.einsum("bhie,bhje->bhij", doh, vh)
    ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
    dq = scale * np.einsum("bhij,bhje->bhie", ds, kh)
    dk = scale * np.einsum("bhij,bhie->bhje", ds, qh)
    return _tokens(dq), _tokens(dk), _tokens(dv)


def rowdot(o, do, B, L, H):
    """D [B, H, L] = sum_e do[i, h, e] o[i, h, e]: equals sum_j p[i, j] dp[i, j]
    (the row term of ds) because o[i] = sum_j p[i, j] v[j]."""
    return np.einsum("bhie,bhie->bhi", _heads(o, B, L, H), _heads(do, B, L, H))
