"""Token-sharded data parallelism on the host: two ranks over gloo (127.0.0.1).

Each rank takes its contiguous share of the token rows (``dp.shard_rows``),
computes that share's weight gradients, writes them into its flat gradient
buffer (``dp.GradBuffer``) and sums the buffers with one all-reduce
(``dp.allreduce_grads``). The summed gradients must equal the gradients of the
whole batch, and each rank's dx its rows of the whole batch's dx -- the fp64
oracle on all the tokens is the reference. The per-rank compute here is the
oracle, so that the test runs without a GPU; the GPU path runs the library's
backward into the same buffer (tests/test_dp_gpu.py).
"""
import json
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

CASES = {
    "full-T11": dict(T=11, d=16, r=4, d_ff=24, S=2),
    "mlp-T10": dict(T=10, d=16, r=4, d_ff=24, S=2, kind="mlp"),
    "dense-T9": dict(T=9, d=16, r=4, d_ff=24, S=2, dense=True),
    "uneven-ranks-T12": dict(T=12, d=16, r=8, d_ff=24, S=2, ranks=(8, 16, 24, 8, 16, 8, 24)),
    "attn-T12-L3": dict(T=12, d=16, r=4, d_ff=24, S=2, attn=True, seq_len=3),
}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle(cfg, inp, lo, hi):
    import oracle as O
    f = {k: v.astype(np.float64) for k, v in inp.items()}
    p = {k: f[k] for k in cfg.param_shapes()}
    oc = dict(kind=cfg.kind, dense=cfg.dense, sigma=cfg.sigma, eps=cfg.eps, attn=cfg.attn,
              seq_len=cfg.seq_len or None, heads=2 if cfg.attn else None)
    x, dy = f["x"][lo:hi], f["dy"][lo:hi]
    full = cfg.kind == "full" and not cfg.attn
    dq = f["dq"][lo:hi] if full else None
    dk = f["dk"][lo:hi] if full else None
    _, saved = O.block_forward(p, x, oc)
    return O.block_backward(p, x, saved, dy, dq, dk, oc)


def _rank_main(rank, world, port, out_dir, name):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank))
    import torch.distributed as dist
    from rank_bottleneck_gb300 import dp
    from rank_bottleneck_gb300.block import BlockConfig
    from rank_bottleneck_gb300.synth import make_block_inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = BlockConfig(dtype="f32", **CASES[name])
    # every rank draws the same seeded batch (weights and tokens) and keeps its rows
    inp = make_block_inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, kind=cfg.kind, dense=cfg.dense,
                            dtype="f32", seed=3, ranks=cfg.ranks)
    if cfg.attn:
        L = cfg.seq_len
        slo, shi = dp.shard_rows(cfg.T // L, rank, world)
        lo, hi = slo * L, shi * L
    else:
        lo, hi = dp.shard_rows(cfg.T, rank, world)
    dx, g = _oracle(cfg, inp, lo, hi)
    buf = dp.GradBuffer(cfg, "cpu", torch.float64)
    for k, v in g.items():
        buf[k].copy_(torch.from_numpy(v))
    dp.allreduce_grads(buf)
    dist.destroy_process_group()
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), lo=lo, hi=hi, dx=dx, values=buf.values,
             **{"g_" + k: v.numpy() for k, v in buf.grads.items()})


@pytest.mark.parametrize("name", list(CASES))
def test_two_token_shards_allreduced_equal_the_whole_batch(tmp_path, name):
    from rank_bottleneck_gb300.block import BlockConfig
    from rank_bottleneck_gb300.synth import make_block_inputs
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path), name), nprocs=world, join=True)
    res = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    cfg = BlockConfig(dtype="f32", **CASES[name])
    inp = make_block_inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, kind=cfg.kind, dense=cfg.dense,
                            dtype="f32", seed=3, ranks=cfg.ranks)
    dx, g = _oracle(cfg, inp, 0, cfg.T)
    # the shards tile the batch
    assert int(res[0]["lo"]) == 0 and int(res[0]["hi"]) == int(res[1]["lo"])
    assert int(res[1]["hi"]) == cfg.T
    for r in res:
        lo, hi = int(r["lo"]), int(r["hi"])
        np.testing.assert_allclose(r["dx"], dx[lo:hi], rtol=1e-12, atol=1e-12)
        for k, v in g.items():
            np.testing.assert_allclose(r["g_" + k], v, rtol=1e-11, atol=1e-12, err_msg=k)
    # one all-reduce carries every weight gradient: sum of r_i (d_in + d_out) + norm weights
    d, dff = cfg.d, cfg.d_ff
    if cfg.dense:
        want = (3 * d * d + d * d if cfg.kind == "full" else 0) + 2 * dff * d + d * dff
    else:
        rq, rk, rv, ro, rg, ru, rd = cfg.layer_ranks()
        want = (rq + rk + rv) * 2 * d + ro * 2 * d if cfg.kind == "full" else 0
        want += (rg + ru) * (d + dff) + rd * (dff + d)
    want += 2 * d if cfg.kind == "full" else d
    assert int(res[0]["values"]) == want


def test_shard_rows_tile_any_batch():
    from rank_bottleneck_gb300.dp import shard_rows
    for T in (1, 7, 16, 16384, 16385):
        for world in (1, 2, 3, 8):
            if T < world:
                continue
            parts = [shard_rows(T, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
            sizes = [hi - lo for lo, hi in parts]
            assert max(sizes) - min(sizes) <= 1


def test_grad_buffer_views_are_aligned_and_cover_the_shapes():
    from rank_bottleneck_gb300.block import BlockConfig
    from rank_bottleneck_gb300.dp import GradBuffer
    cfg = BlockConfig(T=8, d=2048, r=512, d_ff=5461, S=4)
    buf = GradBuffer(cfg, "cpu")
    shapes = cfg.param_shapes()
    assert set(buf.grads) == set(shapes)
    for k, v in buf.grads.items():
        assert tuple(v.shape) == shapes[k]
        assert v.data_ptr() % 16 == 0
        if k == "A_d":
            assert v.stride(0) == cfg.ld_ff
    # the exchange is about 2.5x smaller than the dense block's at r = d/4
    dense = GradBuffer(BlockConfig(T=8, d=4096, r=1024, d_ff=11008, S=8, dense=True), "cpu")
    lowrank = GradBuffer(BlockConfig(T=8, d=4096, r=1024, d_ff=11008, S=8), "cpu")
    assert 2.4 < dense.values / lowrank.values < 2.6
