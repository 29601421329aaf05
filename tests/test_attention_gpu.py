"""Parity of the attention core (tcgen05 kernels, ``include/boostattn.h``)
against the fp64 oracle (``oracle.attention``, pinned in
test_oracle_attention_pins.py), element by element on the same bf16 inputs.

Bars, from the arithmetic: the kernels round p (forward) and p, ds (backward)
to bf16 before they multiply (relative error 2^-9 each, averaging over the
keys) and store o, dq, dk, dv in bf16 (2^-9); everything else accumulates in
fp32. So the worst element may be off by a few bf16 steps of the tensor's
largest value: max |gpu - oracle| <= 2e-2 max |oracle|, and over the tensor
the RMS error <= 1e-2 of the RMS value (scales below 1e-3 count as 1e-3: the
values here are of order 0.1 to 10, and a reference that is exactly zero
leaves only fp32 rounding). lse is fp32 from bf16 inputs:
|gpu - oracle| <= 1e-3.
"""
import numpy as np
import pytest

from oracle import attention as OA

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_bottleneck_gb300 import _build
    _build.build()


def close(got, ref, name, tol=2e-2, rms=1e-2, floor=1e-3):
    """floor: the scale below which a reference counts as zero (a single token's
    dq and dk are exactly 0 in the oracle and fp32 rounding in the kernels)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = max(float(np.max(np.abs(ref))), floor)
    err = float(np.max(np.abs(got - ref)))
    assert err <= tol * scale, f"{name}: max err {err:.3e} vs max {scale:.3e}"
    r = float(np.sqrt(np.mean((got - ref) ** 2)) / max(np.sqrt(np.mean(ref ** 2)), floor))
    assert r <= rms, f"{name}: rms err {r:.3e}"


def run_gpu(B, L, H, causal, seed=0, q_scale=1.0):
    from rank_bottleneck_gb300 import attention as A
    from rank_bottleneck_gb300.synth import make_attention_inputs
    inp = make_attention_inputs(B, L, H, 128, seed=seed, q_scale=q_scale)
    dev = {k: torch.from_numpy(v).to("cuda", torch.bfloat16) for k, v in inp.items()}
    cfg = A.AttnConfig(B=B, L=L, H=H, causal=causal)
    ws = A.AttnWorkspace(cfg)
    o = A.forward(cfg, dev["q"], dev["k"], dev["v"], ws)
    dq, dk, dv = A.backward(cfg, dev["q"], dev["k"], dev["v"], o, dev["do"], ws)
    assert A.device_status(ws) == 0
    out = dict(o=o, dq=dq, dk=dk, dv=dv)
    res = {k: t.float().cpu().numpy() for k, t in out.items()}
    res["lse"] = ws.lse_view(cfg).cpu().numpy()
    res["o_bf16"] = res["o"]
    return inp, res


def oracle(inp, B, L, H, causal):
    f = {k: v.astype(np.float64) for k, v in inp.items()}
    o, lse = OA.attention_forward(f["q"], f["k"], f["v"], B, L, H, causal)
    dq, dk, dv = OA.attention_backward(f["q"], f["k"], f["v"], f["do"], B, L, H, causal)
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


CASES = [
    (1, 128, 1, True),     # one tile, two streamed blocks
    (2, 384, 2, True),     # several tiles per sequence
    (2, 200, 3, True),     # ragged: 200 = 128 + 72, the last block 8 rows
    (1, 320, 2, False),    # non-causal
    (3, 65, 1, False),     # ragged non-causal, one row past a block
    (1, 1, 2, True),       # a single token: o = v
    (2, 129, 1, True),     # one row into the second tile
    (1, 136, 20, True),    # 20 heads: the backward's row terms take each row as a
                           # group of 16 heads and one of 4
]


@pytest.mark.parametrize("B,L,H,causal", CASES)
def test_attention_matches_oracle(B, L, H, causal):
    inp, got = run_gpu(B, L, H, causal, seed=B * 1000 + L)
    ref = oracle(inp, B, L, H, causal)
    for k in ("o", "dq", "dk", "dv"):
        close(got[k], ref[k], k)
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= 1e-3


def test_single_token_is_value():
    inp, got = run_gpu(1, 1, 2, True)
    assert np.array_equal(got["o"], inp["v"])      # p = 1 exactly, v already bf16


def test_sharp_softmax():
    """q scaled by 8: most rows put nearly all weight on one key (large score
    gaps exercise the running-maximum rescale)."""
    inp, got = run_gpu(1, 256, 2, True, seed=7, q_scale=8.0)
    ref = oracle(inp, 1, 256, 2, True)
    for k in ("o", "dq", "dk", "dv"):
        close(got[k], ref[k], k)
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= 1e-2


def test_deterministic():
    _, a = run_gpu(2, 256, 2, True, seed=3)
    _, b = run_gpu(2, 256, 2, True, seed=3)
    for k in ("o", "dq", "dk", "dv", "lse"):
        assert np.array_equal(a[k], b[k]), k


def test_full_size_sampled_heads():
    """The 1B block's attention shape (4 sequences of 4096 tokens, 16 heads of
    128: T = 16384, d = 2048), in the launch configuration the bench times;
    two (sequence, head) slices checked whole against the oracle."""
    B, L, H = 4, 4096, 16
    inp, got = run_gpu(B, L, H, True, seed=11)
    for b, h in ((0, 0), (3, 13)):
        rows = slice(b * L, (b + 1) * L)
        cols = slice(h * 128, (h + 1) * 128)
        sl = {k: v[rows, cols] for k, v in inp.items()}
        ref = oracle(sl, 1, L, 1, True)
        for k in ("o", "dq", "dk", "dv"):
            close(got[k][rows, cols], ref[k], f"{k}[{b},{h}]")
        assert np.max(np.abs(got["lse"][b, h] - ref["lse"][0, 0])) <= 1e-3
