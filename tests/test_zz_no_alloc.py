"""bn_weight_grad_noalloc: the weight-gradient GEMM for callers that cannot
allocate GPU memory (all of their memory is pre-reserved by their own pool, or
an allocation is not allowed where they run). The fp32 partial tiles of its K
split live in a fixed array inside the library instead of in caller scratch.

Each result is checked against an fp64 numpy product of the same bf16 inputs
(the engine tests' bar, 1e-2 of the largest reference value) and against the
entry point that takes caller scratch (bn_testing_gemm, STORE epilogue with K
split). Two calls run in a row, and both cut their left-over tiles along K
(checked from the launch records: each call launches the split reduction), with
different tile counts and split depths, so partial tiles left in the shared
array by the first call would show up in the second. A wait that runs out is
reported by bn_weight_grad_noalloc_status. Runs alone or after the other tests;
it is in its own file, collected last."""
import ctypes
import time

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
    f = lib.bn_weight_grad_noalloc_status
    f.argtypes = [ctypes.c_void_p]
    f.restype = ctypes.c_int
    f = lib.bn_testing_weight_grad_noalloc_unfed
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def draw(rng, shape, scale=1.0):
    """bf16-exact values: the same numbers on the host (fp64) and on the device."""
    a = round_to_bf16((rng.standard_normal(shape) * scale).astype(np.float32))
    return a.astype(np.float64), torch.from_numpy(a).to("cuda", torch.bfloat16)


def stream():
    return torch.cuda.current_stream().cuda_stream


def noalloc(lib, M, N, T, A, B, colv, out):
    return lib.bn_weight_grad_noalloc(M, N, T, A.data_ptr(), A.stride(0), B.data_ptr(),
                                      B.stride(0), None if colv is None else colv.data_ptr(),
                                      out.data_ptr(), out.stride(0), stream())


def with_caller_scratch(lib, M, N, T, A, B, colv, out):
    from _gemmhook import run
    q = dict(M=M, N=N, K=T, a=A, b=B, lda=A.stride(0), ldb=B.stride(0), a_mn=True, b_mn=True,
             out0=out, ldo=out.stride(0), colv=colv)
    run(lib, "store", [q], dtype="bf16", allow_split=True)


def rel(got, ref):
    return float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))


@pytest.mark.parametrize("first, second", [((1024, 1024, 4096), (512, 264, 4000))])
def test_noalloc_two_split_calls_match_fp64_and_caller_scratch(lib, first, second):
    from rank_bottleneck_gb300 import block as Bk
    rng = np.random.default_rng(0)
    for (M, N, T), use_colv in ((first, True), (second, False)):
        a64, A = draw(rng, (T, M))
        b64, B = draw(rng, (T, N), 1 / np.sqrt(T))
        c64, colv = draw(rng, (N,)) if use_colv else (None, None)
        want = a64.T @ b64
        if use_colv:
            want = want * c64[None, :]
        got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        Bk.profile_start()
        st = noalloc(lib, M, N, T, A, B, colv, got)
        recs = Bk.profile_stop()
        assert st == 0, lib.bn_status_string(st)
        assert lib.bn_weight_grad_noalloc_status(stream()) == 0
        kinds = [r["kernel"] for r in recs]
        assert kinds.count("gemm_tcgen05") == 1 and kinds.count("splitk_reduce") == 1, kinds
        g = got.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(g))
        assert rel(g, want) <= TOL
        ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        with_caller_scratch(lib, M, N, T, A, B, colv, ref)
        assert rel(g, ref.float().cpu().numpy().astype(np.float64)) <= TOL


def test_noalloc_large_output(lib):
    """The fixed array bounds the partial tiles per SM, not M x N: a 4608 x 4100
    gradient (whole rounds of tiles plus split left-over tiles) runs; 96 sampled
    rows match fp64 and the whole output matches the caller-scratch entry point."""
    rng = np.random.default_rng(1)
    M, N, T = 4608, 4100, 4096
    a64, A = draw(rng, (T, M))
    b64, Bw = draw(rng, (T, N + 4), 1 / np.sqrt(T))
    B = Bw[:, :N]
    got = torch.full((M, N + 4), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :N]
    st = noalloc(lib, M, N, T, A, B, None, got)
    assert st == 0, lib.bn_status_string(st)
    assert lib.bn_weight_grad_noalloc_status(stream()) == 0
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g))
    rows = np.unique(np.concatenate([[0, 255, 256, M - 1], rng.choice(M, 92, replace=False)]))
    want = a64[:, rows].T @ b64[:, :N]
    assert rel(g[rows], want) <= TOL
    ref = torch.empty(M, N + 4, dtype=torch.bfloat16, device="cuda")[:, :N]
    with_caller_scratch(lib, M, N, T, A, B, None, ref)
    assert rel(g, ref.float().cpu().numpy().astype(np.float64)) <= TOL


def test_noalloc_timeout_is_reported(lib):
    """A launch whose wait can never be satisfied gives up after 1 s; the status
    call reports BN_ERR_TIMEOUT (5) once and then BN_OK, and the next ordinary
    call on the same array is correct."""
    rng = np.random.default_rng(2)
    M, N, T = 256, 256, 128
    a64, A = draw(rng, (T, M))
    b64, B = draw(rng, (T, N))
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    counters = torch.zeros(2, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    st = lib.bn_testing_weight_grad_noalloc_unfed(M, N, T, A.data_ptr(), M, B.data_ptr(), N,
                                                  out.data_ptr(), N, counters.data_ptr(), stream())
    assert st == 0, lib.bn_status_string(st)
    status = lib.bn_weight_grad_noalloc_status(stream())
    waited = time.perf_counter() - t0
    assert lib.bn_status_string(status) == b"BN_ERR_TIMEOUT"
    assert 0.5 < waited < 30.0                        # the 1 s limit, not a hang
    assert torch.all(out == 7.0)                      # nothing was stored
    assert lib.bn_weight_grad_noalloc_status(stream()) == 0   # read and cleared
    st = noalloc(lib, M, N, T, A, B, None, out)
    assert st == 0 and lib.bn_weight_grad_noalloc_status(stream()) == 0
    assert rel(out.float().cpu().numpy().astype(np.float64), a64.T @ b64) <= TOL


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
