"""fp64 CPU oracle for one CoLA-style low-rank bottleneck decoder block.

TEST INFRASTRUCTURE ONLY. This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``. The library (``rank_bottleneck_gb300``) never imports,
links or calls it, and it imports nothing from the library: its inputs arrive
as plain numpy arrays.

What it computes, and where each step comes from ("BOOST" below is the
project page *BOOST: BOttleneck-Optimized Scalable Training Framework for
Low-Rank Large Language Models*; "BOOST-MLSys26" is the paper summary page of
that name):

* bottleneck linear layer  out = B . sigma(A . x), A [r, d_in], B [d_out, r],
  sigma = SiLU (CoLA) or identity (SVD-style)
  -- BOOST, "Move the chunk boundary to the bottleneck", first paragraph.
* one LLaMA decoder block with every linear layer factorised: pre-RMSNorm,
  Q/K/V, O, residual, pre-RMSNorm, gate/up, SwiGLU, down, residual
  -- BOOST, same section, the decoder-block figure and its caption; the layer
  set is fixed by the all-reduce volume table (3r + r + 2r + r = 7r down
  widths, 5d + 2 d_ff up widths). By default the attention core is not part
  of the path and the O projection reads V directly; with cfg["attn"] the
  causal attention core of ``oracle.attention`` runs between them (sequences
  of cfg["seq_len"] tokens, cfg["heads"] heads, d / 128 unless given) and the
  O projection reads its output.
* RMSNorm is the plain definition n = x * w / sqrt(mean(x^2) + eps). Online
  RMSNorm reaches this result exactly -- BOOST, "Three supporting changes" ->
  Online RMSNorm ("gives the exact result"), and BOOST-MLSys26, core method ->
  Online RMSNorm (the correction alpha = RMS_local / RMS_global is
  mathematically equivalent). The literal S-shard emulation is
  ``online_rmsnorm_linear`` below; it exists to pin that claim.
* linear-layer grouping (QKV and gate+up) and low-rank activation
  checkpointing change where the work runs, not what it computes -- BOOST,
  "Three supporting changes" -> Linear layer grouping / Checkpointing without
  communication. The oracle therefore writes each factorised layer on its own
  and, in checkpoint mode, re-runs the same forward helpers from the saved
  pre-activations.
* the pages give no backward pass; the gradients here are the plain
  derivatives of the forward definition above.
* bottlenecks of uneven size: BOOST, Limitations -> "Untested extensions",
  says the design also covers bottlenecks of different sizes. Each factorised
  layer i then has its own rank r_i (A_i [r_i, d_in], B_i [d_out, r_i]); the
  grouped tensors are the layers' slices side by side ([T, r_q + r_k + r_v],
  [T, r_g + r_u]). The oracle reads every r_i off the parameter shapes.

Readings where the pages are silent:
eps = 1e-5 inside the square root of both the local and the global RMS;
SwiGLU m = SiLU(G) * U; sigma on every factorised layer (including the gate
and up bottlenecks, with SwiGLU's own SiLU on G on top); checkpoint mode saves
the pre-activations z (sigma' needs z and SiLU cannot be inverted from h).
Precision: everything in float64; bf16 inputs arrive already rounded and are
never rounded again.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_backward, attention_forward

EPS = 1e-5


# ----------------------------------------------------------------------------
# elementwise pieces
# ----------------------------------------------------------------------------

def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    """SiLU(z) = z * sigmoid(z): the CoLA bottleneck nonlinearity and SwiGLU's gate."""
    return z * sigmoid(z)


def silu_grad(z):
    """d/dz [z * sigmoid(z)] = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def act(z, sigma):
    """The bottleneck nonlinearity: 'silu' (CoLA) or 'identity' (SVD-style)."""
    if sigma == "silu":
        return silu(z)
    if sigma == "identity":
        return z.copy()
    raise ValueError(sigma)


def act_grad(z, sigma):
    if sigma == "silu":
        return silu_grad(z)
    if sigma == "identity":
        return np.ones_like(z)
    raise ValueError(sigma)


# ----------------------------------------------------------------------------
# RMSNorm and its Online (sharded) form
# ----------------------------------------------------------------------------

def rmsnorm(x, w, eps=EPS):
    """Plain RMSNorm over the last axis. Returns (n, rstd) with rstd = 1/rms."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(ms + eps)
    return x * rstd * w, rstd


def rmsnorm_backward(dn, x, w, rstd):
    """Gradient of n = x * w * rstd(x). Returns (dx, dw).

    dw_j = sum_t dn_tj x_tj rstd_t
    dx_tj = rstd_t g_tj - x_tj rstd_t^3 mean_k(g_tk x_tk),   g = dn * w
    """
    dw = np.sum(dn * x * rstd, axis=0)
    g = dn * w
    dx = rstd * g - x * rstd ** 3 * np.mean(g * x, axis=-1, keepdims=True)
    return dx, dw


def shard_bounds(d, S):
    """S contiguous equal column shards of the hidden dimension (d % S == 0)."""
    if S < 1 or d % S:
        raise ValueError(f"d={d} is not split evenly into S={S} shards")
    w = d // S
    return [(s * w, (s + 1) * w) for s in range(S)]


def online_rmsnorm_linear(x, w, A, S, eps=EPS):
    """Online RMSNorm followed by the down-projection, emulated over S shards.

    BOOST, "Three supporting changes" -> Online RMSNorm: each shard normalises
    its slice of the hidden vector by its own (local) RMS and multiplies by its
    slice of the down-projection; the shard's sum of squares travels with the
    partial product; the partial is scaled back by its local RMS and divided by
    the global RMS. BOOST-MLSys26 writes the combined per-row factor as
    alpha = RMS_local / RMS_global.  Returns z = n @ A.T with n = RMSNorm(x).
    """
    T, d = x.shape
    partials, local_rms, sumsq = [], [], []
    for lo, hi in shard_bounds(d, S):
        xs = x[:, lo:hi]
        ss = np.sum(xs * xs, axis=1)                      # shard's sum of squares
        rms_s = np.sqrt(ss / (hi - lo) + eps)             # local RMS
        local = xs * w[lo:hi] / rms_s[:, None]            # locally normalised slice
        partials.append(local @ A[:, lo:hi].T)            # shard's partial product
        local_rms.append(rms_s)
        sumsq.append(ss)
    rms_g = np.sqrt(np.sum(sumsq, axis=0) / d + eps)      # global RMS from the sums
    z = np.zeros((T, A.shape[0]))
    for P_s, rms_s in zip(partials, local_rms):
        alpha = rms_s / rms_g                              # per-row correction
        z += alpha[:, None] * P_s
    return z


# ----------------------------------------------------------------------------
# one bottleneck layer
# ----------------------------------------------------------------------------

def lowrank_forward(X, A, B, sigma):
    """out = sigma(X A^T) B^T for token rows X [T, d_in]. Returns (out, z, h)."""
    z = X @ A.T
    h = act(z, sigma)
    return h @ B.T, z, h


def lowrank_backward(dout, X, z, h, A, B, sigma):
    """Gradients of out = sigma(X A^T) B^T. Returns (dX, dA, dB)."""
    dB = dout.T @ h
    dh = dout @ B
    dz = dh * act_grad(z, sigma)
    dA = dz.T @ X
    dX = dz @ A
    return dX, dA, dB


def swiglu(G, U):
    """m = SiLU(G) * U."""
    return silu(G) * U


def swiglu_backward(dm, G, U):
    return dm * U * silu_grad(G), dm * silu(G)


# ----------------------------------------------------------------------------
# the block
# ----------------------------------------------------------------------------

def _cfg(cfg):
    c = dict(kind="full", dense=False, sigma="silu", eps=EPS, checkpoint=False, attn=False,
             seq_len=None, heads=None)
    c.update(cfg or {})
    if c["dense"] and c["checkpoint"]:
        raise ValueError("low-rank activation checkpointing applies to the factorised block only")
    return c


def _split(a, parts):
    return np.split(a, parts, axis=1)


def _cuts(widths):
    """Column offsets at which a grouped [T, sum(widths)] tensor splits into its
    layers' slices (np.split indices)."""
    return list(np.cumsum(widths)[:-1])


def qkv_ranks(p):
    """Ranks of the grouped Q, K, V bottlenecks, read off their up-projections
    B [d_out, r_i]: each factorised layer may have its own rank."""
    return [p["B_q"].shape[1], p["B_k"].shape[1], p["B_v"].shape[1]]


def gu_ranks(p):
    """Ranks of the grouped gate and up bottlenecks."""
    return [p["B_g"].shape[1], p["B_u"].shape[1]]


def _qkv_up(p, z_qkv, c):
    """h = sigma(z) for the three grouped bottlenecks, then the Q, K, V up-projections."""
    h_qkv = act(z_qkv, c["sigma"])
    h_q, h_k, h_v = _split(h_qkv, _cuts(qkv_ranks(p)))
    return dict(h_qkv=h_qkv, q=h_q @ p["B_q"].T, k=h_k @ p["B_k"].T, v=h_v @ p["B_v"].T)


def _o_up(p, x, z_o, c):
    h_o = act(z_o, c["sigma"])
    return dict(h_o=h_o, x1=x + h_o @ p["B_o"].T)


def _gu_up(p, z_gu, c):
    h_gu = act(z_gu, c["sigma"])
    h_g, h_u = _split(h_gu, _cuts(gu_ranks(p)))
    G = h_g @ p["B_g"].T
    U = h_u @ p["B_u"].T
    return dict(h_gu=h_gu, G=G, U=U, m=swiglu(G, U))


def _down_up(p, x1, z_d, c):
    h_d = act(z_d, c["sigma"])
    return dict(h_d=h_d, y=x1 + h_d @ p["B_d"].T)


def _attn_shape(c, x):
    T, d = x.shape
    L = c["seq_len"]
    H = c["heads"] if c["heads"] else d // 128
    if not L or T % L or d % H:
        raise ValueError("attn needs T % seq_len == 0 and d % heads == 0")
    return T // L, L, H


def _attention(a, c, x):
    """O (and lse) from q, k, v: the attention core, when it is inside the block."""
    Bs, L, H = _attn_shape(c, x)
    a["o"], a["lse"] = attention_forward(a["q"], a["k"], a["v"], Bs, L, H, causal=True)


def block_forward(p, x, cfg=None):
    """Forward of one block. Returns (outputs, saved).

    outputs = {"y": [T, d]} plus {"q", "k": [T, d]} for the full block.
    saved   = every activation the backward reads, or in checkpoint mode only
              the [T, k r] pre-activations z_qkv, z_o, z_gu, z_d.
    """
    c = _cfg(cfg)
    a = {}
    if c["kind"] == "full":
        n1, rstd1 = rmsnorm(x, p["w_norm1"], c["eps"])
        a.update(n1=n1, rstd1=rstd1)
        if c["dense"]:
            qkv = n1 @ p["A_qkv"].T
            q, k, v = _split(qkv, 3)
            a.update(q=q, k=k, v=v)
            if c["attn"]:
                _attention(a, c, x)
            a["x1"] = x + a["o" if c["attn"] else "v"] @ p["A_o"].T
        else:
            a["z_qkv"] = n1 @ p["A_qkv"].T
            a.update(_qkv_up(p, a["z_qkv"], c))
            if c["attn"]:
                _attention(a, c, x)
            a["z_o"] = a["o" if c["attn"] else "v"] @ p["A_o"].T
            a.update(_o_up(p, x, a["z_o"], c))
    elif c["kind"] == "mlp":
        a["x1"] = x
    else:
        raise ValueError(c["kind"])
    n2, rstd2 = rmsnorm(a["x1"], p["w_norm2"], c["eps"])
    a.update(n2=n2, rstd2=rstd2)
    if c["dense"]:
        gu = n2 @ p["A_gu"].T
        G, U = _split(gu, 2)
        a.update(G=G, U=U, m=swiglu(G, U))
        a["y"] = a["x1"] + a["m"] @ p["A_d"].T
    else:
        a["z_gu"] = n2 @ p["A_gu"].T
        a.update(_gu_up(p, a["z_gu"], c))
        a["z_d"] = a["m"] @ p["A_d"].T
        a.update(_down_up(p, a["x1"], a["z_d"], c))
    outputs = {"y": a["y"]}
    if c["kind"] == "full" and not c["attn"]:
        outputs.update(q=a["q"], k=a["k"])
    if c["checkpoint"]:
        keep = ("z_qkv", "z_o", "z_gu", "z_d") if c["kind"] == "full" else ("z_gu", "z_d")
        saved = {key: a[key] for key in keep}
    else:
        saved = a
    return outputs, saved


def recompute(p, x, saved, cfg=None):
    """Rebuild every activation the backward reads from the saved pre-activations.

    BOOST, "Three supporting changes" -> Checkpointing without communication:
    only the r-wide activations are stored and the rest of the chunk is re-run
    in the backward pass. Uses the very same helpers, in the same order, as
    ``block_forward``.
    """
    c = _cfg(cfg)
    a = dict(saved)
    if c["kind"] == "full":
        n1, rstd1 = rmsnorm(x, p["w_norm1"], c["eps"])
        a.update(n1=n1, rstd1=rstd1)
        a.update(_qkv_up(p, a["z_qkv"], c))
        if c["attn"]:
            _attention(a, c, x)
        a.update(_o_up(p, x, a["z_o"], c))
    else:
        a["x1"] = x
    n2, rstd2 = rmsnorm(a["x1"], p["w_norm2"], c["eps"])
    a.update(n2=n2, rstd2=rstd2)
    a.update(_gu_up(p, a["z_gu"], c))
    a.update(_down_up(p, a["x1"], a["z_d"], c))
    return a


def block_backward(p, x, saved, dy, dq=None, dk=None, cfg=None):
    """Backward of one block for upstream gradients dy (and dq, dk; None = 0).

    Returns (dx, grads) with grads keyed like the parameters. Gradients are of
    L = sum(y * dy) + sum(q * dq) + sum(k * dk).
    """
    c = _cfg(cfg)
    a = recompute(p, x, saved, c) if c["checkpoint"] else saved
    s = c["sigma"]
    g = {}
    T = x.shape[0]

    # MLP half: y = x1 + Down(SwiGLU(Gate(n2), Up(n2))), n2 = RMSNorm(x1)
    if c["dense"]:
        g["A_d"] = dy.T @ a["m"]
        dm = dy @ p["A_d"]
        dG, dU = swiglu_backward(dm, a["G"], a["U"])
        dgu = np.concatenate([dG, dU], axis=1)
        g["A_gu"] = dgu.T @ a["n2"]
        dn2 = dgu @ p["A_gu"]
    else:
        dm, g["A_d"], g["B_d"] = lowrank_backward(dy, a["m"], a["z_d"], a["h_d"],
                                                  p["A_d"], p["B_d"], s)
        dG, dU = swiglu_backward(dm, a["G"], a["U"])
        cut = _cuts(gu_ranks(p))
        A_g, A_u = np.split(p["A_gu"], cut, axis=0)
        z_g, z_u = _split(a["z_gu"], cut)
        h_g, h_u = _split(a["h_gu"], cut)
        dn2_g, dA_g, g["B_g"] = lowrank_backward(dG, a["n2"], z_g, h_g, A_g, p["B_g"], s)
        dn2_u, dA_u, g["B_u"] = lowrank_backward(dU, a["n2"], z_u, h_u, A_u, p["B_u"], s)
        g["A_gu"] = np.concatenate([dA_g, dA_u], axis=0)
        dn2 = dn2_g + dn2_u
    dx1_norm, g["w_norm2"] = rmsnorm_backward(dn2, a["x1"], p["w_norm2"], a["rstd2"])
    dx1 = dy + dx1_norm
    if c["kind"] == "mlp":
        return dx1, g

    # attention-projection half: x1 = x + O(V) (or O(attention(Q, K, V))),
    # Q, K, V = projections of n1 = RMSNorm(x)
    dq = np.zeros((T, x.shape[1])) if dq is None else dq
    dk = np.zeros((T, x.shape[1])) if dk is None else dk
    X_o = a["o" if c["attn"] else "v"]

    def core_backward(dX):
        """dV from the O projection's input gradient; with the attention core
        inside, its backward gives dQ, dK, dV (dq, dk from outside are 0)."""
        if not c["attn"]:
            return dq, dk, dX
        Bs, L, H = _attn_shape(c, x)
        return attention_backward(a["q"], a["k"], a["v"], dX, Bs, L, H, causal=True)

    if c["dense"]:
        g["A_o"] = dx1.T @ X_o
        dq, dk, dv = core_backward(dx1 @ p["A_o"])
        dqkv = np.concatenate([dq, dk, dv], axis=1)
        g["A_qkv"] = dqkv.T @ a["n1"]
        dn1 = dqkv @ p["A_qkv"]
    else:
        dX, g["A_o"], g["B_o"] = lowrank_backward(dx1, X_o, a["z_o"], a["h_o"],
                                                  p["A_o"], p["B_o"], s)
        dq, dk, dv = core_backward(dX)
        cut = _cuts(qkv_ranks(p))
        A_q, A_k, A_v = np.split(p["A_qkv"], cut, axis=0)
        z_q, z_k, z_v = _split(a["z_qkv"], cut)
        h_q, h_k, h_v = _split(a["h_qkv"], cut)
        dn1_q, dA_q, g["B_q"] = lowrank_backward(dq, a["n1"], z_q, h_q, A_q, p["B_q"], s)
        dn1_k, dA_k, g["B_k"] = lowrank_backward(dk, a["n1"], z_k, h_k, A_k, p["B_k"], s)
        dn1_v, dA_v, g["B_v"] = lowrank_backward(dv, a["n1"], z_v, h_v, A_v, p["B_v"], s)
        g["A_qkv"] = np.concatenate([dA_q, dA_k, dA_v], axis=0)
        dn1 = dn1_q + dn1_k + dn1_v
    dx_norm, g["w_norm1"] = rmsnorm_backward(dn1, x, p["w_norm1"], a["rstd1"])
    return dx1 + dx_norm, g


def loss(p, x, dy, dq=None, dk=None, cfg=None):
    """L = sum(y * dy) + sum(q * dq) + sum(k * dk): the scalar whose gradient
    ``block_backward`` returns (used by the finite-difference pins)."""
    out, _ = block_forward(p, x, cfg)
    L = np.sum(out["y"] * dy)
    if "q" in out and dq is not None:
        L += np.sum(out["q"] * dq)
    if "k" in out and dk is not None:
        L += np.sum(out["k"] * dk)
    return L
