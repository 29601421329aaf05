"""Pins for the oracle's bottleneck-aware tensor parallelism (BTP) emulation.

BOOST, "Move the chunk boundary to the bottleneck": shifting each tensor
parallel chunk to start at a column-split up-projection and end at a row-split
down-projection changes where partial sums are added, not what the block
computes; each chunk's one all-reduce carries an r-wide activation, 7r values
per token per block and pass (the page's volume table, "BOOST 7bsr").

* the BTP data flow (``oracle.btp``) equals the plain block (``oracle.block``,
  itself pinned in test_oracle_pins.py) for every shard count, shard bounds,
  sigma and block kind, forward and backward;
* the widths of the all-reduces the emulation performs add up to the page's
  closed form: 7r per token and pass (3r for the MLP sub-block alone), and
  7r / 2d = 0.88 of full-rank TP at LLaMA-7B shapes, as printed;
* a planted mistake (one shard's partial dropped from an all-reduce) fails the
  equality by far.
"""
import numpy as np
import pytest

import oracle as O
from oracle import btp
from rank_bottleneck_gb300.synth import make_block_inputs


def inputs(T, d, r, d_ff, kind="full", seed=0):
    a = {k: v.astype(np.float64) for k, v in
         make_block_inputs(T, d, r, d_ff, kind=kind, dtype="f32", seed=seed).items()}
    x, dy = a.pop("x"), a.pop("dy")
    return a, x, dy, a.pop("dq", None), a.pop("dk", None)


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def run_both(p, x, dy, dq, dk, S, cfg, bd=None, bf=None):
    ref, saved = O.block_forward(p, x, cfg)
    rdx, rg = O.block_backward(p, x, saved, dy, dq, dk, cfg)
    out, acts, vf = btp.block_forward_btp(p, x, S, cfg, bd, bf)
    dx, g, vb = btp.block_backward_btp(p, x, acts, dy, S, dq, dk, cfg, bd, bf)
    err = max([rel(out[k], ref[k]) for k in ref] + [rel(dx, rdx)] + [rel(g[k], rg[k]) for k in rg])
    return err, vf, vb


@pytest.mark.parametrize("S", [1, 2, 4, 8])
@pytest.mark.parametrize("sigma", ["silu", "identity"])
@pytest.mark.parametrize("kind", ["full", "mlp"])
def test_btp_equals_plain_block(S, sigma, kind):
    p, x, dy, dq, dk = inputs(T=6, d=32, r=8, d_ff=48, kind=kind, seed=S)
    err, _, _ = run_both(p, x, dy, dq, dk, S, dict(kind=kind, sigma=sigma))
    assert err <= 1e-12


def test_btp_uneven_shard_bounds():
    p, x, dy, dq, dk = inputs(T=5, d=32, r=8, d_ff=45)
    bd = [(0, 5), (5, 16), (16, 32)]
    bf = [(0, 7), (7, 20), (20, 21), (21, 45)]
    # Online RMSNorm takes each shard's own width for its local RMS
    err, _, _ = run_both(p, x, dy, dq, dk, 3, {}, bd, bf)
    assert err <= 1e-12


def test_btp_allreduce_volume_is_7r():
    T, d, r, d_ff = 4, 32, 8, 48
    for kind, per_pass in (("full", 7 * r), ("mlp", 3 * r)):
        p, x, dy, dq, dk = inputs(T, d, r, d_ff, kind=kind)
        _, vf, vb = run_both(p, x, dy, dq, dk, 4, dict(kind=kind))
        assert vf["r_wide"] == per_pass and vb["r_wide"] == per_pass
        # one RMSNorm statistic per token and norm: forward sums of squares,
        # backward row sums of dn * w * x
        norms = 2 if kind == "full" else 1
        assert vf["norm"] == norms and vb["norm"] == norms
    # the page's ratio to full-rank TP (2bsd) at LLaMA-7B shapes: 0.88
    d7, r7 = 4096, 1024
    assert round(7 * r7 / (2 * d7), 2) == 0.88


def test_btp_planted_dropped_partial_fails(monkeypatch):
    p, x, dy, dq, dk = inputs(T=4, d=32, r=8, d_ff=48)
    orig = btp._Comm.allreduce

    def drop_last(self, partials, kind="r"):
        return orig(self, partials[:-1] if kind == "r" else partials, kind)

    monkeypatch.setattr(btp._Comm, "allreduce", drop_last)
    err, _, _ = run_both(p, x, dy, dq, dk, 4, {})
    assert err > 1e-2
