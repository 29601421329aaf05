"""The block with the causal attention core inside (desc.attn = 1) against the
fp64 oracle (``oracle.block`` with cfg["attn"], pinned by finite differences in
test_oracle_pins.py), forward and backward through the C ABI.

The O projection reads O = attention(Q, K, V) instead of V; Q, K never leave
the block, so the only upstream gradient is dy. Bars as for the plain block
(max |gpu - ref| / max |ref| per tensor, 2e-2 for bf16).
"""
import numpy as np
import pytest

import _blockcase as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_bottleneck_gb300 import _build
    _build.build()


def case(kw, seed=0):
    from rank_bottleneck_gb300.block import BlockConfig
    cfg = BlockConfig(**kw)
    inp = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, kind=cfg.kind, dense=cfg.dense,
                   dtype=cfg.dtype, seed=seed)
    return cfg, inp


SMALL = {
    # 2 sequences of 128, 2 heads
    "attn-T256-L128-d256": dict(T=256, d=256, r=64, d_ff=333, S=4, attn=True, seq_len=128),
    # ragged sequences (100 = 64 + 36), 3 of them
    "attn-T300-L100-d256": dict(T=300, d=256, r=64, d_ff=333, S=2, attn=True, seq_len=100),
    "attn-identity": dict(T=256, d=384, r=32, d_ff=200, S=3, sigma="identity", attn=True,
                          seq_len=256),
    "attn-ckpt": dict(T=256, d=256, r=64, d_ff=333, S=4, attn=True, seq_len=128,
                      checkpoint=True),
    "attn-dense": dict(T=256, d=256, r=8, d_ff=344, S=4, dense=True, attn=True, seq_len=128),
    "attn-btp": dict(T=256, d=256, r=64, d_ff=333, S=4, btp=True, attn=True, seq_len=128),
    "attn-L1": dict(T=3, d=128, r=8, d_ff=24, S=2, attn=True, seq_len=1),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_attn_block_matches_oracle(name):
    cfg, inp = case(SMALL[name])
    got = C.run_gpu(cfg, inp)
    assert set(got) >= {"y", "dx"} and "q" not in got
    ref = C.run_oracle(cfg, inp)
    C.compare(got, ref, C.TOL["bf16"])


def test_attn_checkpoint_is_bit_identical():
    kw = dict(T=256, d=256, r=64, d_ff=333, S=4, attn=True, seq_len=128)
    cfg_a, inp = case(kw)
    cfg_b, _ = case(dict(kw, checkpoint=True))
    a = C.run_gpu(cfg_a, inp)
    b = C.run_gpu(cfg_b, inp)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_attn_block_1b_widths():
    """The 1B block's widths (d = 2048: 16 heads, r = 512, d_ff = 5461, S = 4)
    with two sequences of 1024 tokens, every output and gradient compared."""
    cfg, inp = case(dict(T=2048, d=2048, r=512, d_ff=5461, S=4, attn=True, seq_len=1024), seed=4)
    got = C.run_gpu(cfg, inp)
    ref = C.run_oracle(cfg, inp)
    C.compare(got, ref, C.TOL["bf16"])
