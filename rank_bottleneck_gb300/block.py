"""Python binding of libboostblk.so (ctypes). Argument marshalling only: every
step of the block runs in the library's kernels. PyTorch provides device memory
and the current CUDA stream.

    cfg = BlockConfig(T=16384, d=2048, r=512, d_ff=5461, S=4)
    ws = Workspace(cfg, device="cuda")
    out = forward(cfg, params, x, ws)               # {"y", "q", "k"}
    dx, grads = backward(cfg, params, x, ws, dy, dq, dk)

`params` maps the names of ``PARAM_NAMES`` to tensors of the block's dtype;
d_ff-wide tensors (A_d) may be views with a padded row stride (ld_ff).

The library allocates no memory and does not synchronise inside a forward or
backward call, so with every output buffer passed in, both calls can be
captured into a CUDA graph (after one direct call on the device, which sets up
per-device state) and replayed.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

PARAM_NAMES = ("w_norm1", "A_qkv", "B_q", "B_k", "B_v", "A_o", "B_o",
               "w_norm2", "A_gu", "B_g", "B_u", "A_d", "B_d")
ATTN_NAMES = ("w_norm1", "A_qkv", "B_q", "B_k", "B_v", "A_o", "B_o")
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libboostblk.so")

BN_F32, BN_BF16 = 0, 1
SIGMAS = {"identity": 0, "silu": 1}
KINDS = {"full": 0, "mlp": 1}


class _Desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("r", ctypes.c_int64),
                ("d_ff", ctypes.c_int64), ("ld_ff", ctypes.c_int64), ("S", ctypes.c_int32),
                ("sigma", ctypes.c_int32), ("dtype", ctypes.c_int32), ("kind", ctypes.c_int32),
                ("dense", ctypes.c_int32), ("checkpoint", ctypes.c_int32), ("eps", ctypes.c_float),
                ("btp", ctypes.c_int32), ("attn", ctypes.c_int32), ("seq_len", ctypes.c_int32),
                ("r_layer", ctypes.c_int64 * 7)]


class _Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


class LaunchRecord(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("epi", ctypes.c_int32), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double), ("ms", ctypes.c_float)]


KERNEL_NAMES = ("gemm_tcgen05", "gemm_fp32", "splitk_reduce", "norm_stats", "norm_weight_fold",
                "rmsnorm_backward", "dw_colsum", "elementwise", "attention")

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the in-tree library. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with rank_bottleneck_gb300._build.build()")
    lib = ctypes.CDLL(path)
    vp, st = ctypes.c_void_p, ctypes.c_int
    lib.bn_block_workspace_size.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(ctypes.c_size_t),
                                            ctypes.POINTER(ctypes.c_size_t)]
    lib.bn_block_workspace_size.restype = st
    lib.bn_block_forward.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(_Params), vp, vp, vp, vp,
                                     vp, vp, vp]
    lib.bn_block_forward.restype = st
    lib.bn_block_backward.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(_Params), vp, vp, vp,
                                      vp, vp, vp, ctypes.POINTER(_Params), vp, vp]
    lib.bn_block_backward.restype = st
    lib.bn_get_device_status.argtypes = [vp, vp]
    lib.bn_get_device_status.restype = st
    lib.bn_last_launch_count.argtypes = []
    lib.bn_last_launch_count.restype = ctypes.c_int
    lib.bn_status_string.argtypes = [st]
    lib.bn_status_string.restype = ctypes.c_char_p
    lib.bn_last_cuda_error.argtypes = []
    lib.bn_last_cuda_error.restype = ctypes.c_char_p
    lib.bn_profile_start.argtypes = []
    lib.bn_profile_start.restype = st
    lib.bn_profile_stop.argtypes = [ctypes.POINTER(LaunchRecord), ctypes.c_int]
    lib.bn_profile_stop.restype = ctypes.c_int
    _lib = lib
    return lib


@dataclass
class BlockConfig:
    T: int
    d: int
    r: int
    d_ff: int
    ld_ff: int | None = None
    S: int = 1
    sigma: str = "silu"
    dtype: str = "bf16"
    kind: str = "full"
    dense: bool = False
    checkpoint: bool = False
    eps: float = 1e-5
    btp: bool = False  # bottleneck-aware tensor parallelism emulated over the S shards
    attn: bool = False  # the causal attention core inside the block (heads of 128)
    seq_len: int = 0    # tokens per sequence when attn
    # per-layer ranks (q, k, v, o, gate, up, down) for bottlenecks of uneven size;
    # None (or a 0 entry) = r
    ranks: tuple | None = None

    def __post_init__(self):
        if self.ld_ff is None:
            self.ld_ff = (self.d_ff + 63) // 64 * 64  # whole 128-byte rows

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def desc(self) -> _Desc:
        return _Desc(self.T, self.d, self.r, self.d_ff, self.ld_ff, self.S, SIGMAS[self.sigma],
                     BN_BF16 if self.dtype == "bf16" else BN_F32, KINDS[self.kind],
                     int(self.dense), int(self.checkpoint), self.eps, int(self.btp),
                     int(self.attn), int(self.seq_len),
                     (ctypes.c_int64 * 7)(*(self.ranks or (0,) * 7)))

    def layer_ranks(self):
        """(r_q, r_k, r_v, r_o, r_g, r_u, r_d)."""
        return tuple(int(x) if x else self.r for x in (self.ranks or (0,) * 7))

    def param_shapes(self):
        """Logical shape of each parameter (A_d has ld_ff-strided rows)."""
        d, dff = self.d, self.d_ff
        if self.dense:
            s = dict(w_norm1=(d,), A_qkv=(3 * d, d), A_o=(d, d), w_norm2=(d,),
                     A_gu=(2 * dff, d), A_d=(d, dff))
        else:
            rq, rk, rv, ro, rg, ru, rd = self.layer_ranks()
            s = dict(w_norm1=(d,), A_qkv=(rq + rk + rv, d), B_q=(d, rq), B_k=(d, rk),
                     B_v=(d, rv), A_o=(ro, d), B_o=(d, ro), w_norm2=(d,), A_gu=(rg + ru, d),
                     B_g=(dff, rg), B_u=(dff, ru), A_d=(rd, dff), B_d=(d, rd))
        if self.kind == "mlp":
            for n in ATTN_NAMES:
                s.pop(n, None)
        return s


def _check(status: int):
    if status != 0:
        lib = load()
        name = lib.bn_status_string(status).decode()
        raise RuntimeError(f"boostblk: {name} ({lib.bn_last_cuda_error().decode()})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def workspace_size(cfg: BlockConfig):
    saved, scratch = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().bn_block_workspace_size(ctypes.byref(cfg.desc()), ctypes.byref(saved),
                                          ctypes.byref(scratch)))
    return saved.value, scratch.value


class Workspace:
    """Device buffers `saved` and `scratch` for one block (status word zeroed)."""

    def __init__(self, cfg: BlockConfig, device="cuda"):
        n_saved, n_scratch = workspace_size(cfg)
        self.saved = torch.empty(max(n_saved, 16), dtype=torch.uint8, device=device)
        self.scratch = torch.empty(max(n_scratch, 256), dtype=torch.uint8, device=device)
        self.scratch[:256].zero_()


def empty_param(cfg: BlockConfig, name: str, device="cuda"):
    """An uninitialised parameter-shaped tensor (A_d with ld_ff-padded rows)."""
    shape = cfg.param_shapes()[name]
    if name == "A_d":
        return torch.empty(shape[0], cfg.ld_ff, dtype=cfg.torch_dtype, device=device)[:, :cfg.d_ff]
    return torch.empty(shape, dtype=cfg.torch_dtype, device=device)


def _params_struct(cfg: BlockConfig, params) -> _Params:
    p = _Params()
    shapes = cfg.param_shapes()
    for n in PARAM_NAMES:
        t = params.get(n) if params is not None else None
        if n in shapes:
            if t is None:
                raise ValueError(f"missing parameter {n}")
            if tuple(t.shape) != shapes[n] or t.dtype != cfg.torch_dtype:
                raise ValueError(f"{n}: expected {shapes[n]} {cfg.torch_dtype}, got "
                                 f"{tuple(t.shape)} {t.dtype}")
            want_ld = cfg.ld_ff if n == "A_d" else (shapes[n][-1] if len(shapes[n]) == 2 else 1)
            if t.stride(-1) != 1 or (t.dim() == 2 and t.stride(0) != want_ld):
                raise ValueError(f"{n}: rows must be contiguous with leading dimension {want_ld}")
            setattr(p, n, t.data_ptr())
        else:
            setattr(p, n, None)
    return p


def forward(cfg: BlockConfig, params, x, ws: Workspace, y=None, q=None, k=None, stream=None):
    """Forward pass; returns {"y": y} (+ "q", "k" for the full block whose attention
    core runs outside it)."""
    full = cfg.kind == "full" and not cfg.attn
    y = torch.empty_like(x) if y is None else y
    if full:
        q = torch.empty_like(x) if q is None else q
        k = torch.empty_like(x) if k is None else k
    P = _params_struct(cfg, params)
    _check(load().bn_block_forward(ctypes.byref(cfg.desc()), ctypes.byref(P), _ptr(x), _ptr(y),
                                   _ptr(q if full else None), _ptr(k if full else None),
                                   _ptr(ws.saved), _ptr(ws.scratch), _stream(stream)))
    out = {"y": y}
    if full:
        out.update(q=q, k=k)
    return out


def backward(cfg: BlockConfig, params, x, ws: Workspace, dy, dq=None, dk=None, dx=None,
             grads=None, stream=None):
    """Backward pass; returns (dx, grads) with grads keyed like the parameters."""
    dx = torch.empty_like(x) if dx is None else dx
    if grads is None:
        grads = {n: empty_param(cfg, n, x.device) for n in cfg.param_shapes()}
    P = _params_struct(cfg, params)
    G = _params_struct(cfg, grads)
    _check(load().bn_block_backward(ctypes.byref(cfg.desc()), ctypes.byref(P), _ptr(x),
                                    _ptr(ws.saved), _ptr(dy), _ptr(dq), _ptr(dk), _ptr(dx),
                                    ctypes.byref(G), _ptr(ws.scratch), _stream(stream)))
    return dx, grads


def device_status(ws: Workspace, stream=None) -> int:
    """Synchronise and read (then clear) the kernels' status word; 0 = OK, 5 = timeout."""
    return load().bn_get_device_status(_ptr(ws.scratch), _stream(stream))


def last_launch_count() -> int:
    return load().bn_last_launch_count()


def profile_start():
    """Record every kernel the library launches from this thread (CUDA events)."""
    load().bn_profile_start()


def profile_stop(max_records=1 << 16):
    """Stop recording; returns [{"kernel", "epi", "flops", "bytes", "ms"}, ...]."""
    buf = (LaunchRecord * max_records)()
    n = load().bn_profile_stop(buf, max_records)
    return [dict(kernel=KERNEL_NAMES[r.kernel], epi=r.epi, flops=r.flops, bytes=r.bytes, ms=r.ms)
            for r in buf[:min(n, max_records)]]
