"""The block's forward and backward captured into a CUDA graph and replayed.

The library allocates nothing and never synchronises inside bn_block_forward /
bn_block_backward, so a caller may capture both calls once and replay them
(bench.py does, to take the host's launch work out of the step). A replay must
give, bit for bit, what the same calls give when issued directly -- also after
new input values are copied into the captured buffers.
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


@pytest.mark.parametrize("kw", [dict(T=600, d=256, r=64, d_ff=333, S=4),
                                dict(T=512, d=256, r=64, d_ff=333, S=4, attn=True, seq_len=256),
                                dict(T=300, d=256, r=64, d_ff=333, S=4, checkpoint=True)],
                         ids=["plain", "attn", "ckpt"])
def test_graph_replay_equals_direct_calls(kw):
    from rank_bottleneck_gb300 import block as B
    cfg = B.BlockConfig(**kw)
    qk = not cfg.attn
    acts = ("x", "dy") + (("dq", "dk") if qk else ())
    inp0 = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, seed=0)
    # two batches for the same weights: seed 0's, and seed 1's tokens and gradients
    inp1 = dict(inp0)
    other = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, seed=1)
    for n in acts:
        inp1[n] = other[n]
    batches = (inp0, inp1)
    outs = [C.run_gpu(cfg, inp) for inp in batches]   # direct calls, fresh buffers
    # the same block captured once, replayed on the two batches
    params, dev = C.to_device(cfg, inp0)
    ws = B.Workspace(cfg, "cuda")
    y, dx = torch.empty_like(dev["x"]), torch.empty_like(dev["x"])
    q = torch.empty_like(dev["x"]) if qk else None
    k = torch.empty_like(dev["x"]) if qk else None
    grads = {n: B.empty_param(cfg, n, "cuda") for n in cfg.param_shapes()}
    dq, dk = (dev["dq"], dev["dk"]) if qk else (None, None)

    def step():
        B.forward(cfg, params, dev["x"], ws, y, q, k)
        B.backward(cfg, params, dev["x"], ws, dev["dy"], dq, dk, dx, grads)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                               # first call outside capture (per-device setup)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed, (inp, want) in enumerate(zip(batches, outs)):
        for n in acts:
            dev[n].copy_(torch.from_numpy(inp[n]).to("cuda", dev[n].dtype))
        g.replay()
        torch.cuda.synchronize()
        assert B.device_status(ws) == 0
        got = {"y": y, "dx": dx, **{"d" + n: t for n, t in grads.items()}}
        if qk:
            got.update(q=q, k=k)
        for name, t in got.items():
            assert np.array_equal(t.float().cpu().numpy().astype(np.float64), want[name]), (seed, name)
