"""bn_weight_grad_noalloc: the weight-gradient GEMM for callers that cannot
allocate GPU memory (all of their memory is pre-reserved by their own pool, or
an allocation is not allowed where they run). The fp32 partial tiles of its K
split live in a fixed array inside the library instead of in caller scratch.

Checked against the entry point that takes caller scratch (bn_testing_gemm,
STORE epilogue with K split) on two calls in a row -- a large problem and then a
smaller one, so stale partial tiles left in the shared array by the first call
would show up in the second. Runs alone or after the other tests; it is in its
own file, collected last."""
import ctypes

import numpy as np
import pytest

from rank_bottleneck_gb300.synth import round_to_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-2  # the bf16 bar of the GEMM engine tests


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_bottleneck_gb300 import _build
    _build.build()
    from rank_bottleneck_gb300 import block as B
    lib = B.load()
    f = lib.bn_weight_grad_noalloc
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def bf16(rng, shape, scale=1.0):
    return torch.from_numpy(round_to_bf16((rng.standard_normal(shape) * scale)
                                          .astype(np.float32))).to("cuda", torch.bfloat16)


def noalloc(lib, M, N, T, A, B, colv, out):
    st = lib.bn_weight_grad_noalloc(M, N, T, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                    None if colv is None else colv.data_ptr(), out.data_ptr(),
                                    out.stride(0), torch.cuda.current_stream().cuda_stream)
    return st


def with_caller_scratch(lib, M, N, T, A, B, colv, out):
    from _gemmhook import run
    q = dict(M=M, N=N, K=T, a=A, b=B, lda=A.stride(0), ldb=B.stride(0), a_mn=True, b_mn=True,
             out0=out, ldo=out.stride(0), colv=colv)
    run(lib, "store", [q], dtype="bf16", allow_split=True)


@pytest.mark.parametrize("first, second", [((1536, 2048, 16384), (512, 264, 4000))])
def test_noalloc_matches_caller_scratch_two_calls(lib, first, second):
    rng = np.random.default_rng(0)
    for (M, N, T), use_colv in ((first, True), (second, False)):
        A = bf16(rng, (T, M))
        B = bf16(rng, (T, N), 1 / np.sqrt(T))
        colv = bf16(rng, (N,)) if use_colv else None
        ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        with_caller_scratch(lib, M, N, T, A, B, colv, ref)
        got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = noalloc(lib, M, N, T, A, B, colv, got)
        torch.cuda.synchronize()
        assert st == 0, lib.bn_status_string(st)
        g, r = got.float(), ref.float()
        assert torch.isfinite(g).all()
        e = ((g - r).abs().max() / r.abs().max()).item()
        assert e <= TOL, e


def test_noalloc_large_output(lib):
    """The fixed array bounds the partial tiles per SM, not M x N: a 4608 x 4100
    gradient (whole rounds of tiles plus split left-over tiles) runs and matches
    the caller-scratch entry point."""
    rng = np.random.default_rng(1)
    M, N, T = 4608, 4100, 4096
    A = bf16(rng, (T, M))
    B = bf16(rng, (T, N + 4), 1 / np.sqrt(T))[:, :N]
    ref = torch.empty(M, N + 4, dtype=torch.bfloat16, device="cuda")[:, :N]
    with_caller_scratch(lib, M, N, T, A, B, None, ref)
    got = torch.full((M, N + 4), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :N]
    st = noalloc(lib, M, N, T, A, B, None, got)
    torch.cuda.synchronize()
    assert st == 0, lib.bn_status_string(st)
    g, r = got.float(), ref.float()
    assert torch.isfinite(g).all()
    assert ((g - r).abs().max() / r.abs().max()).item() <= TOL


def test_noalloc_rejects_bad_arguments(lib):
    A = torch.empty(64, 8192, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(64, 8192, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(64, 8192, dtype=torch.bfloat16, device="cuda")
    st = lib.bn_weight_grad_noalloc(0, 8, 8, A.data_ptr(), 8, B.data_ptr(), 8, None,
                                    out.data_ptr(), 8, None)
    assert lib.bn_status_string(st) == b"BN_ERR_INVALID_ARG"
    st = lib.bn_weight_grad_noalloc(8, 8, 8, A.data_ptr() + 2, 8192, B.data_ptr(), 8192, None,
                                    out.data_ptr(), 8192, None)
    assert lib.bn_status_string(st) == b"BN_ERR_ALIGNMENT"
