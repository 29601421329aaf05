"""Bottleneck-aware tensor parallelism (BTP), emulated over S shards in fp64.

TEST INFRASTRUCTURE ONLY, like ``oracle/block.py``: imported by ``tests/``
only; the library never imports it and it imports nothing from the library.

BOOST ("BOOST: BOttleneck-Optimized Scalable Training Framework for Low-Rank
Large Language Models"), "Move the chunk boundary to the bottleneck": a tensor
parallel chunk starts at an up-projection split by columns (each of S shards
owns a slice of its d_out outputs) and ends at the next down-projection split
by rows (each shard owns a slice of its d_in inputs and produces an r-wide
partial product); one all-reduce of the r-wide partials closes the chunk. Per
decoder block and pass the all-reduces carry 3r + r + 2r + r = 7r values per
token (the page's volume table: BOOST 7bsr; with bottlenecks of uneven size,
the sum of the seven ranks). The RMSNorms fall inside chunks
and use Online RMSNorm ("Three supporting changes" -> Online RMSNorm), whose
shard statistics ride on the chunk's all-reduce; grouping makes the Q/K/V (and
gate/up) all-reduces one each ("Linear layer grouping").

This module writes that data flow out literally: every activation between two
all-reduces exists only as per-shard column slices, every down-projection is a
sum over shards of slice products, and ``_Comm`` counts what each all-reduce
carries. It must reach exactly (up to fp64 rounding) what the plain block of
``oracle/block.py`` computes.

Readings where the pages are silent:
* the backward is the plain derivative of the same layout: a column-parallel
  up-projection's input gradient is an r-wide all-reduce of per-shard partials,
  a row-parallel down-projection's input gradient is local;
* the RMSNorm backward needs each row's sum over all d of dn * w * x: a
  one-value-per-token all-reduce per norm, counted apart from the r-wide ones;
* shard bounds of d and d_ff are contiguous slices given by the caller (equal
  by default); any bounds give the same result.
"""
from __future__ import annotations

import numpy as np

from .block import EPS, act, act_grad, gu_ranks, qkv_ranks, silu, silu_grad


def _cuts(widths):
    """np.split offsets of a grouped tensor made of slices of these widths."""
    return list(np.cumsum(widths)[:-1])


def even_bounds(n, S):
    """S contiguous equal slices of range(n) (n % S == 0)."""
    if S < 1 or n % S:
        raise ValueError(f"{n} is not split evenly into {S} shards")
    w = n // S
    return [(s * w, (s + 1) * w) for s in range(S)]


class _Comm:
    """Counts the values per token each emulated all-reduce carries."""

    def __init__(self):
        self.r_wide = 0     # the bottleneck all-reduces (the page's volume)
        self.norm = 0       # RMSNorm statistics: forward sums of squares, backward row sums

    def allreduce(self, partials, kind="r"):
        out = np.zeros_like(partials[0])
        for p in partials:          # shard order
            out = out + p
        if kind == "r":
            self.r_wide += out.shape[1]
        else:
            self.norm += out.shape[1]
        return out


def _slices(a, bounds):
    return [a[:, lo:hi] for lo, hi in bounds]


def _cat(parts):
    return np.concatenate(parts, axis=1)


def _online_norm_down(x_s, w, A, bounds, eps, comm):
    """Online RMSNorm of the sharded x, then the row-parallel down-projection A
    [k, d]: each shard normalises by its local RMS and multiplies its slice; the
    partials and the shard sums of squares go through one all-reduce; alpha =
    RMS_local / RMS_global corrects each partial. Returns (z, n_s, rstd)."""
    d = bounds[-1][1]
    ss = [np.sum(xs * xs, axis=1) for xs in x_s]
    rms_loc = [np.sqrt(v / (hi - lo) + eps) for v, (lo, hi) in zip(ss, bounds)]
    partials = []
    for xs, rl, (lo, hi) in zip(x_s, rms_loc, bounds):
        partials.append((xs * w[lo:hi] / rl[:, None]) @ A[:, lo:hi].T)
    # the sums of squares ride with the partials (one value per token, counted
    # apart from the r-wide part)
    tot = comm.allreduce([v[:, None] for v in ss], kind="norm")[:, 0]
    rms_g = np.sqrt(tot / d + eps)
    scaled = [(rl / rms_g)[:, None] * P for P, rl in zip(partials, rms_loc)]
    z = comm.allreduce(scaled)
    rstd = (1.0 / rms_g)[:, None]
    n_s = [xs * rstd * w[lo:hi] for xs, (lo, hi) in zip(x_s, bounds)]
    return z, n_s, rstd


def _row_down(X_s, A, bounds, comm):
    """Row-parallel down-projection: z = sum_s X_s A[:, s]^T, one all-reduce."""
    return comm.allreduce([Xs @ A[:, lo:hi].T for Xs, (lo, hi) in zip(X_s, bounds)])


def _col_up(h, B, bounds):
    """Column-parallel up-projection: each shard computes its output slice."""
    return [h @ B[lo:hi, :].T for lo, hi in bounds]


def block_forward_btp(p, x, S, cfg=None, bounds_d=None, bounds_ff=None):
    """Forward of the block in the BTP layout over S shards.

    Returns (outputs, acts, volume) with outputs like ``block.block_forward``
    (full arrays, the shards concatenated), acts the per-shard activations the
    backward reads, and volume = {"r_wide": values per token of the r-wide
    all-reduces}.
    """
    c = dict(kind="full", sigma="silu", eps=EPS)
    c.update(cfg or {})
    T, d = x.shape
    d_ff = p["A_d"].shape[1]
    bd = bounds_d or even_bounds(d, S)
    bf = bounds_ff or even_bounds(d_ff, S)
    comm = _Comm()
    a = {"x_s": _slices(x, bd)}
    if c["kind"] == "full":
        a["z_qkv"], a["n1_s"], a["rstd1"] = _online_norm_down(a["x_s"], p["w_norm1"], p["A_qkv"],
                                                              bd, c["eps"], comm)
        a["h_qkv"] = act(a["z_qkv"], c["sigma"])
        h_q, h_k, h_v = np.split(a["h_qkv"], _cuts(qkv_ranks(p)), axis=1)
        a["q_s"] = _col_up(h_q, p["B_q"], bd)
        a["k_s"] = _col_up(h_k, p["B_k"], bd)
        a["v_s"] = _col_up(h_v, p["B_v"], bd)
        a["z_o"] = _row_down(a["v_s"], p["A_o"], bd, comm)
        a["h_o"] = act(a["z_o"], c["sigma"])
        o_s = _col_up(a["h_o"], p["B_o"], bd)
        a["x1_s"] = [xs + os_ for xs, os_ in zip(a["x_s"], o_s)]
    else:
        a["x1_s"] = a["x_s"]
    a["z_gu"], a["n2_s"], a["rstd2"] = _online_norm_down(a["x1_s"], p["w_norm2"], p["A_gu"], bd,
                                                         c["eps"], comm)
    a["h_gu"] = act(a["z_gu"], c["sigma"])
    h_g, h_u = np.split(a["h_gu"], _cuts(gu_ranks(p)), axis=1)
    a["G_s"] = _col_up(h_g, p["B_g"], bf)
    a["U_s"] = _col_up(h_u, p["B_u"], bf)
    a["m_s"] = [silu(G) * U for G, U in zip(a["G_s"], a["U_s"])]      # SwiGLU, shard-local
    a["z_d"] = _row_down(a["m_s"], p["A_d"], bf, comm)
    a["h_d"] = act(a["z_d"], c["sigma"])
    y_s = [x1 + o for x1, o in zip(a["x1_s"], _col_up(a["h_d"], p["B_d"], bd))]
    outputs = {"y": _cat(y_s)}
    if c["kind"] == "full":
        outputs.update(q=_cat(a["q_s"]), k=_cat(a["k_s"]))
    return outputs, a, {"r_wide": comm.r_wide, "norm": comm.norm}


def _col_up_backward(dY_s, h, B, bounds, comm):
    """Backward of a column-parallel up-projection Y_s = h B_s^T: the input
    gradient dh = sum_s dY_s B_s is an r-wide all-reduce; dB_s = dY_s^T h."""
    dh = comm.allreduce([dY @ B[lo:hi, :] for dY, (lo, hi) in zip(dY_s, bounds)])
    dB = np.concatenate([dY.T @ h for dY in dY_s], axis=0)
    return dh, dB


def _row_down_backward(dz, X_s, A, bounds):
    """Backward of a row-parallel down-projection z = sum_s X_s A_s^T: the input
    gradient of each shard is local, dX_s = dz A_s; dA_s = dz^T X_s."""
    dX_s = [dz @ A[:, lo:hi] for lo, hi in bounds]
    dA = np.concatenate([dz.T @ Xs for Xs in X_s], axis=1)
    return dX_s, dA


def _norm_backward(dn_s, x_s, w, rstd, bounds, comm):
    """Sharded RMSNorm backward: the row sum of dn * w * x over all of d is a
    one-value-per-token all-reduce; the rest is shard-local."""
    d = bounds[-1][1]
    row = comm.allreduce([np.sum(dn * w[lo:hi] * xs, axis=1, keepdims=True)
                          for dn, xs, (lo, hi) in zip(dn_s, x_s, bounds)], kind="norm")
    dx_s = [rstd * dn * w[lo:hi] - xs * rstd ** 3 * row / d
            for dn, xs, (lo, hi) in zip(dn_s, x_s, bounds)]
    dw = np.concatenate([np.sum(dn * xs * rstd, axis=0) for dn, xs in zip(dn_s, x_s)])
    return dx_s, dw


def block_backward_btp(p, x, acts, dy, S, dq=None, dk=None, cfg=None, bounds_d=None,
                       bounds_ff=None):
    """Backward of the BTP-layout block. Returns (dx, grads, volume)."""
    c = dict(kind="full", sigma="silu", eps=EPS)
    c.update(cfg or {})
    T, d = x.shape
    d_ff = p["A_d"].shape[1]
    bd = bounds_d or even_bounds(d, S)
    bf = bounds_ff or even_bounds(d_ff, S)
    comm = _Comm()
    a, s, g = acts, c["sigma"], {}
    dy_s = _slices(dy, bd)

    # down bottleneck: y_s = x1_s + h_d B_d,s^T ; z_d = sum_s m_s A_d,s^T
    dh_d, g["B_d"] = _col_up_backward(dy_s, a["h_d"], p["B_d"], bd, comm)
    dz_d = dh_d * act_grad(a["z_d"], s)
    dm_s, g["A_d"] = _row_down_backward(dz_d, a["m_s"], p["A_d"], bf)
    dG_s = [dm * U * silu_grad(G) for dm, G, U in zip(dm_s, a["G_s"], a["U_s"])]
    dU_s = [dm * silu(G) for dm, G in zip(dm_s, a["G_s"])]
    # gate / up bottlenecks (grouped: one 2r-wide all-reduce)
    h_g, h_u = np.split(a["h_gu"], _cuts(gu_ranks(p)), axis=1)
    dh_g = [dG @ p["B_g"][lo:hi, :] for dG, (lo, hi) in zip(dG_s, bf)]
    dh_u = [dU @ p["B_u"][lo:hi, :] for dU, (lo, hi) in zip(dU_s, bf)]
    dh_gu = comm.allreduce([np.concatenate([gp, up], axis=1) for gp, up in zip(dh_g, dh_u)])
    g["B_g"] = np.concatenate([dG.T @ h_g for dG in dG_s], axis=0)
    g["B_u"] = np.concatenate([dU.T @ h_u for dU in dU_s], axis=0)
    dz_gu = dh_gu * act_grad(a["z_gu"], s)
    dn2_s, g["A_gu"] = _row_down_backward(dz_gu, a["n2_s"], p["A_gu"], bd)
    dx1n_s, g["w_norm2"] = _norm_backward(dn2_s, a["x1_s"], p["w_norm2"], a["rstd2"], bd, comm)
    dx1_s = [dyv + dn for dyv, dn in zip(dy_s, dx1n_s)]
    if c["kind"] == "mlp":
        return _cat(dx1_s), g, {"r_wide": comm.r_wide, "norm": comm.norm}

    # O bottleneck: x1_s = x_s + h_o B_o,s^T ; z_o = sum_s v_s A_o,s^T
    dh_o, g["B_o"] = _col_up_backward(dx1_s, a["h_o"], p["B_o"], bd, comm)
    dz_o = dh_o * act_grad(a["z_o"], s)
    dv_s, g["A_o"] = _row_down_backward(dz_o, a["v_s"], p["A_o"], bd)
    # Q / K / V bottlenecks (grouped: one 3r-wide all-reduce)
    dq_s = _slices(np.zeros((T, d)) if dq is None else dq, bd)
    dk_s = _slices(np.zeros((T, d)) if dk is None else dk, bd)
    h_q, h_k, h_v = np.split(a["h_qkv"], _cuts(qkv_ranks(p)), axis=1)
    parts = [np.concatenate([dqs @ p["B_q"][lo:hi, :], dks @ p["B_k"][lo:hi, :],
                             dvs @ p["B_v"][lo:hi, :]], axis=1)
             for dqs, dks, dvs, (lo, hi) in zip(dq_s, dk_s, dv_s, bd)]
    dh_qkv = comm.allreduce(parts)
    g["B_q"] = np.concatenate([v.T @ h_q for v in dq_s], axis=0)
    g["B_k"] = np.concatenate([v.T @ h_k for v in dk_s], axis=0)
    g["B_v"] = np.concatenate([v.T @ h_v for v in dv_s], axis=0)
    dz_qkv = dh_qkv * act_grad(a["z_qkv"], s)
    dn1_s, g["A_qkv"] = _row_down_backward(dz_qkv, a["n1_s"], p["A_qkv"], bd)
    dxn_s, g["w_norm1"] = _norm_backward(dn1_s, a["x_s"], p["w_norm1"], a["rstd1"], bd, comm)
    dx = _cat([a_ + b_ for a_, b_ in zip(dx1_s, dxn_s)])
    return dx, g, {"r_wide": comm.r_wide, "norm": comm.norm}
