"""Python binding of the attention core of libboostblk.so (C ABI in
``include/boostattn.h``). Argument marshalling only: the forward and backward
run in the library's tcgen05 kernels.

    cfg = AttnConfig(B=4, L=4096, H=16)            # d_head = 128, causal
    ws = AttnWorkspace(cfg, device="cuda")
    o = forward(cfg, q, k, v, ws)                  # q, k, v: bf16 [B L, H 128]
    dq, dk, dv = backward(cfg, q, k, v, o, dout, ws)
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import block as _blk


class _AttnDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("L", ctypes.c_int64), ("H", ctypes.c_int64),
                ("d_head", ctypes.c_int64), ("causal", ctypes.c_int32)]


def _lib():
    lib = _blk.load()
    if not getattr(lib, "_attn_bound", False):
        vp, st = ctypes.c_void_p, ctypes.c_int
        lib.bn_attn_lse_stride.argtypes = [ctypes.c_int64]
        lib.bn_attn_lse_stride.restype = ctypes.c_int64
        lib.bn_attn_workspace_size.argtypes = [ctypes.POINTER(_AttnDesc),
                                               ctypes.POINTER(ctypes.c_size_t),
                                               ctypes.POINTER(ctypes.c_size_t)]
        lib.bn_attn_workspace_size.restype = st
        lib.bn_attn_forward.argtypes = [ctypes.POINTER(_AttnDesc), vp, vp, vp, vp, vp, vp, vp]
        lib.bn_attn_forward.restype = st
        lib.bn_attn_backward.argtypes = [ctypes.POINTER(_AttnDesc)] + [vp] * 11
        lib.bn_attn_backward.restype = st
        lib._attn_bound = True
    return lib


@dataclass
class AttnConfig:
    B: int
    L: int
    H: int
    d_head: int = 128
    causal: bool = True

    def desc(self) -> _AttnDesc:
        return _AttnDesc(self.B, self.L, self.H, self.d_head, int(self.causal))

    @property
    def lse_stride(self) -> int:
        return _lib().bn_attn_lse_stride(self.L)


def workspace_size(cfg: AttnConfig):
    """(lse bytes, scratch bytes)."""
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _blk._check(_lib().bn_attn_workspace_size(ctypes.byref(cfg.desc()), ctypes.byref(a),
                                              ctypes.byref(b)))
    return a.value, b.value


class AttnWorkspace:
    """lse [B H, Lp] fp32 and the scratch buffer (status word zeroed)."""

    def __init__(self, cfg: AttnConfig, device="cuda"):
        n_lse, n_scratch = workspace_size(cfg)
        self.lse = torch.empty(n_lse // 4, dtype=torch.float32, device=device)
        self.scratch = torch.empty(n_scratch, dtype=torch.uint8, device=device)
        self.scratch[:256].zero_()

    def lse_view(self, cfg: AttnConfig):
        """lse as [B, H, L] (the padding columns dropped)."""
        return self.lse.view(cfg.B, cfg.H, cfg.lse_stride)[:, :, :cfg.L]


def _check_tokens(cfg: AttnConfig, *ts):
    for t in ts:
        if t is None:
            continue
        if tuple(t.shape) != (cfg.B * cfg.L, cfg.H * cfg.d_head) or t.dtype != torch.bfloat16:
            raise ValueError(f"expected bf16 [{cfg.B * cfg.L}, {cfg.H * cfg.d_head}], got "
                             f"{t.dtype} {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError("attention tensors must be contiguous")


def forward(cfg: AttnConfig, q, k, v, ws: AttnWorkspace, o=None, stream=None):
    """o = softmax(q k^T / sqrt(d_head) [+ causal mask]) v per head; lse into ws.lse."""
    o = torch.empty_like(q) if o is None else o
    _check_tokens(cfg, q, k, v, o)
    P = _blk._ptr
    _blk._check(_lib().bn_attn_forward(ctypes.byref(cfg.desc()), P(q), P(k), P(v), P(o),
                                       P(ws.lse), P(ws.scratch), _blk._stream(stream)))
    return o


def backward(cfg: AttnConfig, q, k, v, o, dout, ws: AttnWorkspace, dq=None, dk=None, dv=None,
             stream=None):
    """(dq, dk, dv) for the upstream gradient dout, from the forward's o and ws.lse."""
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tokens(cfg, q, k, v, o, dout, dq, dk, dv)
    P = _blk._ptr
    _blk._check(_lib().bn_attn_backward(ctypes.byref(cfg.desc()), P(q), P(k), P(v), P(o),
                                        P(ws.lse), P(dout), P(dq), P(dk), P(dv), P(ws.scratch),
                                        _blk._stream(stream)))
    return dq, dk, dv


def device_status(ws: AttnWorkspace, stream=None) -> int:
    """Synchronise and read (then clear) the kernels' status word; 0 = OK, 5 = timeout."""
    return _lib().bn_get_device_status(_blk._ptr(ws.scratch), _blk._stream(stream))
