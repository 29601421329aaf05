"""Bottleneck-aware tensor parallelism emulated over S shards (btp = 1) on the
GPU, against the oracle's BTP data flow (``oracle.btp``, pinned to the plain
block in test_oracle_btp_pins.py).

In btp mode every row-parallel down-projection and every up-projection's input
gradient sums S per-shard partial products in its epilogue: the emulated
r-wide all-reduce (BOOST page, "Move the chunk boundary to the bottleneck").
The oracle runs the same data flow with the GPU's shard bounds: d in S equal
slices, d_ff in S runs of whole 64-column blocks (tensor-core engine) or of
single columns (fp32 engine). Bars as for the plain block: 2e-2 bf16, 1e-5 fp32.
"""
import numpy as np
import pytest

import _blockcase as C
from oracle import btp as OB

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_bottleneck_gb300 import _build
    _build.build()


def cfg_of(**kw):
    from rank_bottleneck_gb300.block import BlockConfig
    return BlockConfig(**kw)


def ff_bounds(d_ff, S, dtype):
    """The d_ff shards of the GPU: runs of whole k-blocks (64 columns) for bf16,
    of columns for fp32."""
    unit = 64 if dtype == "bf16" else 1
    nb = -(-d_ff // unit)
    return [(unit * (s * nb // S), min(d_ff, unit * ((s + 1) * nb // S))) for s in range(S)]


def run_oracle_btp(cfg, inp, rows=None):
    f = {k: v.astype(np.float64) for k, v in inp.items()}
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    x, dy = sel(f["x"]), sel(f["dy"])
    dq = sel(f["dq"]) if "dq" in f else None
    dk = sel(f["dk"]) if "dk" in f else None
    p = {k: f[k] for k in cfg.param_shapes()}
    oc = dict(kind=cfg.kind, sigma=cfg.sigma, eps=cfg.eps)
    bd = OB.even_bounds(cfg.d, cfg.S)
    bf = ff_bounds(cfg.d_ff, cfg.S, cfg.dtype)
    out, acts, vol_f = OB.block_forward_btp(p, x, cfg.S, oc, bd, bf)
    dx, g, vol_b = OB.block_backward_btp(p, x, acts, dy, cfg.S, dq, dk, oc, bd, bf)
    ranks = cfg.layer_ranks()
    per_pass = sum(ranks) if cfg.kind == "full" else sum(ranks[4:])
    assert vol_f["r_wide"] == per_pass and vol_b["r_wide"] == per_pass
    res = dict(out)
    res["dx"] = dx
    res.update({"d" + k: v for k, v in g.items()})
    return res


SMALL = {
    "full-bf16-S4-ragged": dict(T=300, d=256, r=64, d_ff=333, S=4, btp=True),
    "full-bf16-S8-identity": dict(T=256, d=512, r=128, d_ff=1000, S=8, sigma="identity", btp=True),
    "mlp-bf16-S2": dict(T=200, d=256, r=64, d_ff=688, S=2, kind="mlp", btp=True),
    "full-bf16-S3-r8": dict(T=129, d=192, r=8, d_ff=200, S=3, btp=True),
    "full-f32-S4": dict(T=77, d=128, r=32, d_ff=200, S=4, dtype="f32", btp=True),
    "mlp-f32-S4": dict(T=256, d=256, r=64, d_ff=688, S=4, dtype="f32", kind="mlp", btp=True),
    # bottlenecks of uneven size: the r-wide all-reduces carry sum(r_i) per token
    "full-bf16-S4-uneven": dict(T=300, d=256, r=64, d_ff=333, S=4, btp=True,
                                ranks=(64, 32, 96, 40, 72, 24, 56)),
    "full-f32-S4-uneven": dict(T=77, d=128, r=32, d_ff=200, S=4, dtype="f32", btp=True,
                               ranks=(8, 16, 24, 40, 32, 16, 48)),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_btp_block_matches_oracle(name):
    kw = SMALL[name]
    cfg = cfg_of(**kw)
    inp = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, kind=cfg.kind, dtype=cfg.dtype, ranks=cfg.ranks)
    got = C.run_gpu(cfg, inp)
    C.compare(got, run_oracle_btp(cfg, inp), C.TOL[cfg.dtype])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_btp_close_to_plain_layout(dtype):
    """The shard sums change only the order of the additions."""
    kw = dict(T=300, d=256, r=64, d_ff=333, S=4, dtype=dtype)
    cfg = cfg_of(**kw)
    inp = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, dtype=dtype)
    a = C.run_gpu(cfg, inp)
    b = C.run_gpu(cfg_of(**dict(kw, btp=True)), inp)
    for k in a:
        assert C.rel_err(b[k], a[k]) <= C.TOL[dtype], k


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_btp_checkpoint_is_bit_identical(dtype):
    kw = dict(T=300, d=256, r=64, d_ff=333, S=4, dtype=dtype, btp=True)
    cfg = cfg_of(**kw)
    inp = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, dtype=dtype)
    a = C.run_gpu(cfg, inp)
    b = C.run_gpu(cfg_of(**dict(kw, checkpoint=True)), inp)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_btp_full_size_1b():
    """The 1B shape (T 16384, d 2048, r 512, d_ff 5461, S 4) in btp mode, upstream
    gradients kept on sampled rows (as in test_block_parity_gpu.py)."""
    kw = dict(T=16384, d=2048, r=512, d_ff=5461, S=4, btp=True)
    cfg = cfg_of(**kw)
    inp = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 8192, cfg.T - 1],
                                     rng.choice(cfg.T, size=42, replace=False)]))
    keep = np.zeros(cfg.T, dtype=bool)
    keep[rows] = True
    for k in ("dy", "dq", "dk"):
        inp[k][~keep] = 0.0
    got = C.run_gpu(cfg, inp)
    C.compare(got, run_oracle_btp(cfg, inp, rows=rows), C.TOL["bf16"], rows=rows)
