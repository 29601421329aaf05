"""Named workloads (synthetic LLaMA-2-shaped blocks) and the FLOP model used to
report throughput. Shapes follow the project page's LLaMA-2 family with r = d/4
("Move the chunk boundary to the bottleneck": the paper uses r = d/4)."""
from __future__ import annotations

WORKLOADS = {
    # tiny fp32 MLP sub-block, correctness scale
    "mlp-f32-T256-d256-r64-dff688": dict(T=256, d=256, r=64, d_ff=688, S=4, dtype="f32", kind="mlp"),
    # 1B shape: micro-batch 4 x sequence 4096
    "1b-T16384-d2048-r512-dff5461": dict(T=16384, d=2048, r=512, d_ff=5461, S=4),
    # the 1B block at a quarter of the tokens: small enough for multi-pass profiler
    # captures, its d_ff-wide activations still larger than L2
    "1b-T4096-d2048-r512-dff5461": dict(T=4096, d=2048, r=512, d_ff=5461, S=4),
    "7b-T16384-d4096-r1024-dff11008": dict(T=16384, d=4096, r=1024, d_ff=11008, S=8),
    "13b-ckpt-T16384-d5120-r1280-dff13824": dict(T=16384, d=5120, r=1280, d_ff=13824, S=8,
                                                  checkpoint=True),
    # the 1B block with checkpointing at a quarter of the tokens: profiler captures
    # of the recompute kernels
    "1b-ckpt-T4096-d2048-r512-dff5461": dict(T=4096, d=2048, r=512, d_ff=5461, S=4,
                                             checkpoint=True),
    "13b-T16384-d5120-r1280-dff13824": dict(T=16384, d=5120, r=1280, d_ff=13824, S=8),
    # bottleneck-aware tensor parallelism emulated over the S shards: every
    # down-projection and up-projection input gradient sums S partials (the
    # chunk's r-wide all-reduce) in its epilogue
    "1b-btp-T16384-d2048-r512-dff5461": dict(T=16384, d=2048, r=512, d_ff=5461, S=4, btp=True),
    "7b-btp-T16384-d4096-r1024-dff11008": dict(T=16384, d=4096, r=1024, d_ff=11008, S=8,
                                               btp=True),
    # the whole decoder layer: the causal attention core (heads of 128) between the
    # Q/K/V up-projection and the O projection, 4 sequences of 4096 tokens
    "1b-attn-T16384-L4096-d2048-r512-dff5461": dict(T=16384, d=2048, r=512, d_ff=5461, S=4,
                                                    attn=True, seq_len=4096),
    "7b-attn-T16384-L4096-d4096-r1024-dff11008": dict(T=16384, d=4096, r=1024, d_ff=11008, S=8,
                                                      attn=True, seq_len=4096),
    # one sequence of the 1B layer: small enough for multi-pass profiler captures
    "1b-attn-T4096-L4096-d2048-r512-dff5461": dict(T=4096, d=2048, r=512, d_ff=5461, S=4,
                                                   attn=True, seq_len=4096),
}
for _T in (4096, 16384, 32768):
    for _r in (256, 512, 1024, 2048):
        for _s in ("identity", "silu"):
            WORKLOADS[f"sweep-{_s}-T{_T}-r{_r}"] = dict(T=_T, d=4096, r=_r, d_ff=11008, S=8, sigma=_s)
    WORKLOADS[f"sweep-dense-T{_T}"] = dict(T=_T, d=4096, r=1024, d_ff=11008, S=8, dense=True)

DEFAULT = "1b-T16384-d2048-r512-dff5461"


def layers(cfg):
    """(d_in, d_out) of every linear layer of the block."""
    d, dff = cfg.d, cfg.d_ff
    mlp = [(d, dff), (d, dff), (dff, d)]
    attn = [(d, d)] * 4
    return (attn + mlp) if cfg.kind == "full" else mlp


def attn_pairs(cfg) -> float:
    """Visible (query, key) pairs of the causal attention core, over all heads."""
    if not getattr(cfg, "attn", False):
        return 0.0
    L = cfg.seq_len
    return float(cfg.T // L) * (cfg.d // 128) * L * (L + 1) / 2


def model_flops(cfg) -> float:
    """Forward + backward FLOPs of the block's matrix multiplies: 6 T r (d_in + d_out)
    per factorised layer, 6 T d_in d_out per dense layer, and, with the attention
    core inside, 12 x 128 per visible (query, key) pair and head (forward q.k and
    p v; backward dv, dp, dq, dk)."""
    T, r = cfg.T, cfg.r
    core = 12.0 * 128 * attn_pairs(cfg)
    if cfg.dense:
        return float(sum(6 * T * a * b for a, b in layers(cfg))) + core
    return float(sum(6 * T * r * (a + b) for a, b in layers(cfg))) + core


def recompute_flops(cfg) -> float:
    """Work beyond the model FLOPs: the attention backward recomputes q.k twice and
    do.v once (6 x 128 per visible pair and head); checkpoint mode re-runs the V,
    O, gate and up up-projections (2 T r d_out each; also Q and K and the attention
    forward when the core is inside)."""
    extra = 6.0 * 128 * attn_pairs(cfg)
    if not cfg.checkpoint:
        return extra
    T, r = cfg.T, cfg.r
    outs = ([cfg.d, cfg.d] if cfg.kind == "full" else []) + [cfg.d_ff, cfg.d_ff]
    if getattr(cfg, "attn", False):
        outs += [cfg.d, cfg.d]
        extra += 4.0 * 128 * attn_pairs(cfg)
    return extra + float(sum(2 * T * r * o for o in outs))
