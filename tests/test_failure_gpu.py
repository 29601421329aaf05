"""Failure detection on the GPU without a fault: a kernel whose wait can never
be satisfied gives up after its time limit, reports a timeout through the
status word, and leaves the context usable.

The GEMM engine's chained consumer waits for an upstream launch to count its
CTAs (the chained launches of the block); ``bn_testing_gemm_unfed`` launches
one with a counter that nothing increments. Its operand producer's bounded
wait expires after 1 s, every role unwinds, TMEM is freed and the kernel
returns; ``bn_get_device_status`` then reports BN_ERR_TIMEOUT (5), and an
ordinary launch right after it on the same context computes the right result.
"""
import ctypes
import time

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import _gemmhook as H


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_bottleneck_gb300 import _build
    _build.build()
    from rank_bottleneck_gb300 import block as B
    return B.load()


def test_unfed_consumer_times_out_and_context_survives(lib):
    M, N, K = 256, 256, 128
    g = torch.Generator(device="cuda").manual_seed(0)
    a = torch.randn(M, K, device="cuda", generator=g).bfloat16()
    b = torch.randn(N, K, device="cuda", generator=g).bfloat16()
    out = torch.full((M, N), 7.0, device="cuda", dtype=torch.bfloat16)
    counters = torch.zeros(2, dtype=torch.int32, device="cuda")
    scratch = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    prob = H.Problem(M, N, K, a.data_ptr(), None, K, 0, b.data_ptr(), None, K, 0,
                     out.data_ptr(), None, None, N, None, None, N, None, None)
    fn = lib.bn_testing_gemm_unfed
    fn.argtypes = [ctypes.POINTER(H.Problem), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    assert fn(ctypes.byref(prob), counters.data_ptr(), scratch.data_ptr(), scratch.numel(),
              stream.cuda_stream) == 0
    status = lib.bn_get_device_status(ctypes.c_void_p(scratch.data_ptr()),
                                      ctypes.c_void_p(stream.cuda_stream))
    waited = time.perf_counter() - t0
    assert status == 5, lib.bn_status_string(status)           # BN_ERR_TIMEOUT
    assert 0.5 < waited < 30.0                                  # the 1 s limit, not a hang
    assert int(counters[0].item()) == 0
    assert torch.all(out == 7.0)                                # nothing was stored
    # the context is intact: the same problem, launched normally
    out2 = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    H.run(lib, "store", [dict(M=M, N=N, K=K, a=a, b=b, lda=K, ldb=K, out0=out2)], dtype="bf16")
    ref = a.float() @ b.float().T
    err = (out2.float() - ref).abs().max() / ref.abs().max()
    assert err < 1e-2


def test_attention_unfed_times_out_and_context_survives(lib):
    """The attention forward with its first query tile never loaded: its MMA
    thread's wait gives up after 1 s, every role unwinds, the status word reads
    BN_ERR_TIMEOUT, and an ordinary forward right after it matches the oracle."""
    import numpy as np
    from oracle import attention as OA
    from rank_bottleneck_gb300 import attention as A
    from rank_bottleneck_gb300.synth import make_attention_inputs
    B, L, H = 1, 256, 2
    cfg = A.AttnConfig(B=B, L=L, H=H)
    ws = A.AttnWorkspace(cfg)
    inp = make_attention_inputs(B, L, H, 128, seed=5)
    dev = {n: torch.from_numpy(a).to("cuda", torch.bfloat16) for n, a in inp.items()}
    o = torch.zeros_like(dev["q"])
    fn = lib.bn_testing_attn_forward_unfed
    fn.argtypes = [ctypes.POINTER(A._AttnDesc)] + [ctypes.c_void_p] * 7
    fn.restype = ctypes.c_int
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    assert fn(ctypes.byref(cfg.desc()), dev["q"].data_ptr(), dev["k"].data_ptr(),
              dev["v"].data_ptr(), o.data_ptr(), ws.lse.data_ptr(), ws.scratch.data_ptr(),
              stream.cuda_stream) == 0
    status = A.device_status(ws)
    waited = time.perf_counter() - t0
    assert status == 5, lib.bn_status_string(status)           # BN_ERR_TIMEOUT
    assert 0.5 < waited < 30.0
    assert torch.all(o == 0)                                    # nothing was stored
    # the context is intact: the same forward, launched normally
    o = A.forward(cfg, dev["q"], dev["k"], dev["v"], ws)
    assert A.device_status(ws) == 0
    f = {n: a.astype(np.float64) for n, a in inp.items()}
    ref, _ = OA.attention_forward(f["q"], f["k"], f["v"], B, L, H, True)
    err = np.max(np.abs(o.float().cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert err < 2e-2
