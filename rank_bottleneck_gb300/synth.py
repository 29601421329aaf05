"""Seeded synthetic inputs for the low-rank bottleneck decoder block and its
attention core.

This module only draws random numbers and rounds them to the storage precision.
It holds none of the block's arithmetic, so both the CUDA path and the fp64 CPU
oracle can be fed from it without sharing any compute code.

Recipe (one numpy ``Generator(PCG64(seed))`` per call, float32 draws, fixed order):

    x, w_norm1, A_qkv, B_q, B_k, B_v, A_o, B_o, w_norm2, A_gu, B_g, B_u, A_d, B_d, dy, dq, dk

* x, dy, dq, dk ~ N(0, 1)
* RMSNorm weights w = 1 + 0.1 * N(0, 1)
* every factor (and every dense weight) ~ N(0, 1/fan_in), with fan_in the
  width of the input the factor multiplies: d for down-projections that read the
  hidden state, d_ff for the MLP down factor A_d, and r for every up-projection B.
* bottlenecks of uneven size: each factorised layer may have its own rank
  (q, k, v, o, gate, up, down); the grouped factors stack their layers' rows
  (A_qkv [r_q + r_k + r_v, d], A_gu [r_g + r_u, d]).
* the MLP-only kind skips the attention-half tensors (w_norm1 .. B_o, dq, dk);
  the dense (full-rank) kind draws W_qkv [3d, d], W_o [d, d], W_gu [2 d_ff, d],
  W_d [d, d_ff] into the A_* slots and no B_* tensors.
* bf16 runs round every drawn tensor to bf16 (round to nearest even) here, so
  the GPU and the oracle see bit-identical input values.
"""
from __future__ import annotations

import numpy as np

PARAM_ORDER = ("w_norm1", "A_qkv", "B_q", "B_k", "B_v", "A_o", "B_o",
               "w_norm2", "A_gu", "B_g", "B_u", "A_d", "B_d")
ATTN_HALF = ("w_norm1", "A_qkv", "B_q", "B_k", "B_v", "A_o", "B_o")


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even), kept as float32."""
    a32 = np.ascontiguousarray(a, dtype=np.float32)
    u = a32.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


LAYERS = ("q", "k", "v", "o", "g", "u", "d")  # the factorised layers, in rank order


def layer_ranks(r, ranks=None):
    """The seven per-layer ranks (q, k, v, o, gate, up, down): all r, or `ranks`
    where it gives one (0 or None = r)."""
    if ranks is None:
        return (r,) * 7
    if len(ranks) != 7:
        raise ValueError("ranks needs one entry per factorised layer (q, k, v, o, g, u, d)")
    return tuple(int(x) if x else r for x in ranks)


def tensor_shapes(T, d, r, d_ff, kind="full", dense=False, ranks=None):
    """Ordered (name, shape, fan_in or None) for every drawn tensor of one block.
    `ranks` gives each factorised layer its own rank (see layer_ranks)."""
    rq, rk, rv, ro, rg, ru, rd = layer_ranks(r, ranks)
    out = [("x", (T, d), None)]
    if kind == "full":
        out.append(("w_norm1", (d,), "norm"))
        if dense:
            out += [("A_qkv", (3 * d, d), d), ("A_o", (d, d), d)]
        else:
            out += [("A_qkv", (rq + rk + rv, d), d), ("B_q", (d, rq), rq), ("B_k", (d, rk), rk),
                    ("B_v", (d, rv), rv), ("A_o", (ro, d), d), ("B_o", (d, ro), ro)]
    out.append(("w_norm2", (d,), "norm"))
    if dense:
        out += [("A_gu", (2 * d_ff, d), d), ("A_d", (d, d_ff), d_ff)]
    else:
        out += [("A_gu", (rg + ru, d), d), ("B_g", (d_ff, rg), rg), ("B_u", (d_ff, ru), ru),
                ("A_d", (rd, d_ff), d_ff), ("B_d", (d, rd), rd)]
    out.append(("dy", (T, d), None))
    if kind == "full":
        out += [("dq", (T, d), None), ("dk", (T, d), None)]
    return out


def make_block_inputs(T, d, r, d_ff, *, kind="full", dense=False, dtype="bf16", seed=0,
                      ranks=None):
    """Draw every input of one block fwd+bwd. Returns {name: float32 ndarray}."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    for name, shape, fan in tensor_shapes(T, d, r, d_ff, kind, dense, ranks):
        v = rng.standard_normal(shape, dtype=np.float32)
        if fan == "norm":
            v = np.float32(1.0) + np.float32(0.1) * v
        elif fan is not None:
            v *= np.float32(1.0 / np.sqrt(fan))
        if dtype == "bf16":
            v = round_to_bf16(v)
        out[name] = v
    return out


def make_attention_inputs(B, L, H, d_head, *, seed=0, q_scale=1.0):
    """Draw q, k, v and the upstream gradient do of the attention core, each
    [B * L, H * d_head] ~ N(0, 1) (q times q_scale: larger values sharpen the
    softmax), rounded to bf16. Returns {name: float32 ndarray}."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    for name in ("q", "k", "v", "do"):
        v = rng.standard_normal((B * L, H * d_head), dtype=np.float32)
        if name == "q":
            v *= np.float32(q_scale)
        out[name] = round_to_bf16(v)
    return out
