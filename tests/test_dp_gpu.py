"""The data-parallel step on the GPU: the library's backward writes the weight
gradients into the flat buffer (dp.GradBuffer) that the all-reduce sums, through
a one-rank NCCL process group. With one rank the sum is the identity, so the
gradients must equal, bit for bit, those of the plain backward into separately
allocated tensors; and the two token shards of a batch, run one after the
other on this GPU and summed on the host, must match the oracle on the whole
batch (the exchange itself is tested with two gloo ranks in test_dp_cpu.py)."""
import os
import socket

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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_one_rank_nccl_step_equals_plain_backward():
    import torch.distributed as dist
    from rank_bottleneck_gb300 import block as B
    from rank_bottleneck_gb300 import dp
    cfg = B.BlockConfig(T=512, d=256, r=64, d_ff=333, S=4)
    inp = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff)
    params, dev = C.to_device(cfg, inp)
    ref = C.run_gpu(cfg, inp)
    store = dist.TCPStore("127.0.0.1", _free_port(), 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        step = dp.DataParallelBlock(cfg, 0, 1, "cuda")
        out = step.forward(params, dev["x"])
        dx = step.backward(params, dev["x"], dev["dy"], dev["dq"], dev["dk"])
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert np.array_equal(out["y"].float().cpu().numpy(), ref["y"])
    assert np.array_equal(dx.float().cpu().numpy(), ref["dx"])
    for k, v in step.grads.items():
        assert np.array_equal(v.float().cpu().numpy(), ref["d" + k]), k


def test_two_shards_summed_match_the_whole_batch():
    from rank_bottleneck_gb300 import block as B
    from rank_bottleneck_gb300 import dp
    cfg = B.BlockConfig(T=600, d=256, r=64, d_ff=333, S=4, ranks=(64, 32, 96, 40, 72, 24, 56))
    inp = C.inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, ranks=cfg.ranks)
    params, dev = C.to_device(cfg, inp)
    total, dxs = None, []
    for rank in range(2):
        step = dp.DataParallelBlock(cfg, rank, 2, "cuda")   # no process group: no exchange
        lo, hi = step.lo, step.hi
        step.forward(params, dev["x"][lo:hi])
        dxs.append(step.backward(params, dev["x"][lo:hi], dev["dy"][lo:hi], dev["dq"][lo:hi],
                                 dev["dk"][lo:hi]).float())
        g = step.buf.flat.float().clone()
        total = g if total is None else total + g
    torch.cuda.synchronize()
    buf = dp.GradBuffer(cfg, "cuda", torch.float32)
    buf.flat.copy_(total)
    got = {"d" + k: v.cpu().numpy().astype(np.float64) for k, v in buf.grads.items()}
    got["dx"] = torch.cat(dxs).cpu().numpy().astype(np.float64)
    ref = C.run_oracle(cfg, inp)
    C.compare(got, ref, C.TOL["bf16"], keys=list(got))
