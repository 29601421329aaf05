"""fp64 CPU oracle for the low-rank bottleneck block (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this package; the library never does.
"""
from .block import (EPS, act, act_grad, block_backward, block_forward, loss,
                    lowrank_backward, lowrank_forward, online_rmsnorm_linear,
                    recompute, rmsnorm, rmsnorm_backward, shard_bounds, silu,
                    silu_grad, swiglu, swiglu_backward)
