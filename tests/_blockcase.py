"""Shared test plumbing: one seeded block case run through the library (GPU)
and through the fp64 oracle (CPU), compared tensor by tensor.

Error metric (one number per tensor): max |gpu - ref| / max |ref|. Bars:
1e-5 for fp32 blocks, 2e-2 for bf16 blocks (fp32 accumulate).
"""
from __future__ import annotations

import numpy as np

import oracle as O
from rank_bottleneck_gb300.synth import make_block_inputs

TOL = {"f32": 1e-5, "bf16": 2e-2}


def inputs(T, d, r, d_ff, *, kind="full", dense=False, dtype="bf16", seed=0, ranks=None):
    return make_block_inputs(T, d, r, d_ff, kind=kind, dense=dense, dtype=dtype, seed=seed,
                             ranks=ranks)


def oracle_cfg(cfg):
    return dict(kind=cfg.kind, dense=cfg.dense, sigma=cfg.sigma, eps=cfg.eps,
                checkpoint=cfg.checkpoint, attn=cfg.attn, seq_len=cfg.seq_len or None)


def run_oracle(cfg, inp, rows=None):
    """Oracle forward + backward, optionally on a subset of token rows (the
    block is row-independent, so rows of the result depend only on those rows)."""
    f = {k: v.astype(np.float64) for k, v in inp.items()}
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    x, dy = sel(f["x"]), sel(f["dy"])
    dq = sel(f["dq"]) if "dq" in f and not cfg.attn else None
    dk = sel(f["dk"]) if "dk" in f and not cfg.attn else None
    p = {k: f[k] for k in cfg.param_shapes()}
    oc = oracle_cfg(cfg)
    out, saved = O.block_forward(p, x, oc)
    dx, g = O.block_backward(p, x, saved, dy, dq, dk, oc)
    res = dict(out)
    res["dx"] = dx
    res.update({"d" + k: v for k, v in g.items()})
    return res


def to_device(cfg, inp, device="cuda"):
    import torch
    from rank_bottleneck_gb300 import block as B

    dt = cfg.torch_dtype

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)

    params = {}
    for name in cfg.param_shapes():
        if name == "A_d":
            pad = B.empty_param(cfg, "A_d", device)
            pad.copy_(t(inp["A_d"]))
            params[name] = pad
        else:
            params[name] = t(inp[name])
    dev = dict(x=t(inp["x"]), dy=t(inp["dy"]))
    dev["dq"] = t(inp["dq"]) if "dq" in inp else None
    dev["dk"] = t(inp["dk"]) if "dk" in inp else None
    return params, dev


ROW_TENSORS = ("y", "q", "k", "dx")


def run_gpu(cfg, inp, device="cuda", drop_dq=False, drop_dk=False, ws=None, rows=None):
    """Block forward + backward through the C ABI; every result as an fp64 numpy
    array. With `rows`, the token-row outputs (y, q, k, dx) come back on those
    rows only (the weight gradients whole)."""
    import torch
    from rank_bottleneck_gb300 import block as B

    params, dev = to_device(cfg, inp, device)
    ws = B.Workspace(cfg, device) if ws is None else ws
    out = B.forward(cfg, params, dev["x"], ws)
    # with the attention core inside the block, q and k never leave it
    dq = None if (drop_dq or cfg.attn) else dev["dq"]
    dk = None if (drop_dk or cfg.attn) else dev["dk"]
    dx, grads = B.backward(cfg, params, dev["x"], ws, dev["dy"], dq, dk)
    status = B.device_status(ws)
    assert status == 0, f"device status {status}"
    res = {k: v for k, v in out.items()}
    res["dx"] = dx
    res.update({"d" + k: v for k, v in grads.items()})
    torch.cuda.synchronize()
    if rows is not None:
        idx = torch.from_numpy(np.asarray(rows)).to(device)
        res = {k: (v.index_select(0, idx) if k in ROW_TENSORS else v) for k, v in res.items()}
    return {k: v.float().cpu().numpy().astype(np.float64) for k, v in res.items()}


def rel_err(got, ref):
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def compare(got, ref, tol, rows=None, keys=None):
    """Return {name: error} and assert every tensor is within tol. With `rows`,
    the token-row outputs of `got` are whole and compared on those rows."""
    errs = {}
    for k in (keys or ref.keys()):
        g = got[k]
        if rows is not None and k in ROW_TENSORS:
            g = g[rows]
        assert g.shape == ref[k].shape, (k, g.shape, ref[k].shape)
        assert np.all(np.isfinite(g)), k
        errs[k] = rel_err(g, ref[k])
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, f"over tolerance {tol}: {bad} (all: {errs})"
    return errs
