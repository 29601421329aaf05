"""Token-sharded data parallelism for the block: one process per GPU, each with
all the weights and its own token rows, and one all-reduce of the weight
gradients per step.

BOOST project page, "Data and pipeline parallelism need no change": data
parallelism composes with the low-rank block unchanged, and the gradients it
all-reduces are those of the factors (A_i, B_i) and the norm weights -- about
2.5x fewer values than the dense block's at r = d/4. The block is
row-independent in the forward, so rank j's rows need nothing from the other
ranks; the backward's only cross-rank step is the sum of the weight gradients.

Every weight gradient of a step lives in one flat buffer (``GradBuffer``: each
parameter's gradient is a view into it, written in place by the backward), so
the exchange is a single collective over contiguous memory. The collective is
torch.distributed's all-reduce (NCCL on GPUs, gloo on the host); nothing else
crosses ranks.
"""
from __future__ import annotations

from dataclasses import replace

import torch

from . import block as B


def shard_rows(T: int, rank: int, world: int):
    """Contiguous token rows [lo, hi) of `rank` out of `world`: sizes differ by
    at most one row, lower ranks first."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    base, extra = divmod(T, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


class GradBuffer:
    """The weight gradients of one block as views into one flat tensor.

    Each gradient has the parameter's logical shape (A_d with ld_ff-strided
    rows, as the library stores it); every view starts on a 16-byte boundary.
    ``flat`` is what the all-reduce sums; padding between views is zero and
    stays zero under a sum.
    """

    def __init__(self, cfg: B.BlockConfig, device="cuda", dtype=None):
        dtype = cfg.torch_dtype if dtype is None else dtype
        esize = torch.empty(0, dtype=dtype).element_size()
        align = max(1, 16 // esize)
        shapes = cfg.param_shapes()
        layout, off = [], 0
        for name in B.PARAM_NAMES:
            if name not in shapes:
                continue
            shape = shapes[name]
            rows = shape[0] if len(shape) == 2 else 1
            ld = (cfg.ld_ff if name == "A_d" else shape[-1]) if len(shape) == 2 else shape[0]
            layout.append((name, off, shape, ld))
            off += -(-(rows * ld) // align) * align
        self.flat = torch.zeros(off, dtype=dtype, device=device)
        self.grads = {}
        for name, o, shape, ld in layout:
            if len(shape) == 2:
                v = self.flat[o:o + shape[0] * ld].view(shape[0], ld)[:, :shape[1]]
            else:
                v = self.flat[o:o + shape[0]]
            self.grads[name] = v
        self.values = sum(v.numel() for v in self.grads.values())

    def __getitem__(self, name):
        return self.grads[name]


def allreduce_grads(buf: GradBuffer, group=None) -> None:
    """Sum every rank's weight gradients in place (one collective). A no-op
    without an initialised process group of more than one rank."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return
    if dist.get_world_size(group) == 1:
        return
    dist.all_reduce(buf.flat, op=dist.ReduceOp.SUM, group=group)


class DataParallelBlock:
    """One rank's share of a data-parallel block step on `T_global` tokens.

        dp = DataParallelBlock(cfg_global, rank, world, device)
        out = dp.forward(params, x_local)                # y (q, k) for the local rows
        dx = dp.backward(params, x_local, dy_local, dq_local, dk_local)
        dp.grads                                         # summed over all ranks

    ``cfg_global.T`` is the whole batch; this rank runs the library's forward
    and backward on its rows ``shard_rows(T, rank, world)`` and then sums the
    weight gradients over the ranks. With the attention core inside the block,
    shards hold whole sequences (the global T split into sequences of seq_len,
    dealt out like rows).
    """

    def __init__(self, cfg_global: B.BlockConfig, rank: int, world: int, device="cuda",
                 group=None):
        self.rank, self.world, self.group = rank, world, group
        if cfg_global.attn:
            L = cfg_global.seq_len
            lo, hi = shard_rows(cfg_global.T // L, rank, world)
            self.lo, self.hi = lo * L, hi * L
        else:
            self.lo, self.hi = shard_rows(cfg_global.T, rank, world)
        if self.hi <= self.lo:
            raise ValueError(f"rank {rank} of {world} has no token rows")
        self.cfg = replace(cfg_global, T=self.hi - self.lo)
        self.ws = B.Workspace(self.cfg, device)
        self.buf = GradBuffer(self.cfg, device)

    @property
    def grads(self):
        return self.buf.grads

    def forward(self, params, x, y=None, q=None, k=None, stream=None):
        return B.forward(self.cfg, params, x, self.ws, y, q, k, stream)

    def backward(self, params, x, dy, dq=None, dk=None, dx=None, stream=None):
        dx, _ = B.backward(self.cfg, params, x, self.ws, dy, dq, dk, dx, self.buf.grads, stream)
        allreduce_grads(self.buf, self.group)
        return dx
