"""The block's RMSNorm backward on its own (bn_testing_norm_bwd), against the
oracle's `rmsnorm_backward`, and its failure detection.

The kernel takes dn' = rstd * dn (the block's dX GEMM epilogue folds the row's
1/rms in) and adds the residual gradient:
    dx = dres + rstd dn w - x rstd^3 mean(dn w x),   dw = sum_t rstd dn x,
which is the oracle's (dx, dw) for dn = dn' / rstd, plus dres. Widths: 2048
(rows streamed through shared memory, one 256-column chunk per lane and
step, the weights in registers), 320 (a ragged last chunk: lanes past the row
hold nothing), 1024, 2056 (9 chunks on the 12-chunk instance, the weights in
shared memory), 3072, 4096 (16 chunks, four warps a block), 4104 and 5120
(the 13B width: each row split between the two warps of a pair, the second
warp's last chunks past the row at 4104), and 5128 (the two-pass kernel for
wider rows); 1000 rows over the GPU's blocks leave every block a different row
count.

Failure detection: with `unfed` the first row of the kernel's first warp is
never loaded; its bounded wait gives up after 1 s, the status word reads
BN_ERR_TIMEOUT, and the same launch right after it on the same context is
correct again.
"""
import ctypes
import time

import numpy as np
import pytest

import _blockcase as C
import oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_bottleneck_gb300 import _build
    _build.build()
    from rank_bottleneck_gb300 import block as B
    L = B.load()
    L.bn_testing_norm_bwd.argtypes = [ctypes.c_int64, ctypes.c_int64] + [ctypes.c_void_p] * 8 + [
        ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    L.bn_testing_norm_bwd.restype = ctypes.c_int
    return L


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def case(rows, d, seed):
    g = np.random.default_rng(seed)
    x = bf16(g.standard_normal((rows, d))).double().numpy()
    w = bf16(1.0 + 0.1 * g.standard_normal(d)).double().numpy()
    dres = bf16(g.standard_normal((rows, d))).double().numpy()
    _, rstd = O.rmsnorm(x, w)
    rstd32 = rstd.astype(np.float32)                  # what the forward saved
    dnp = bf16(rstd32 * g.standard_normal((rows, d))).double().numpy()   # rstd * dn, bf16
    dx_ref, dw_ref = O.rmsnorm_backward(dnp / rstd32.astype(np.float64), x, w,
                                        rstd32.astype(np.float64))
    return x, w, dres, rstd32, dnp, dx_ref + dres, dw_ref


def launch(lib, x, w, dres, rstd, dnp, unfed=0, scratch=None):
    rows, d = x.shape
    dev = "cuda"
    t = {n: bf16(a).to(dev) for n, a in (("x", x), ("w", w), ("dres", dres), ("dn", dnp))}
    rs = torch.from_numpy(rstd.reshape(-1)).to(dev)
    dx = torch.empty(rows, d, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(d, dtype=torch.bfloat16, device=dev)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    part = torch.empty(2 * sms * d, dtype=torch.float32, device=dev)
    if scratch is None:
        scratch = torch.zeros(256, dtype=torch.uint8, device=dev)
    st = lib.bn_testing_norm_bwd(rows, d, t["dn"].data_ptr(), t["x"].data_ptr(),
                                 t["w"].data_ptr(), rs.data_ptr(), t["dres"].data_ptr(),
                                 dx.data_ptr(), dw.data_ptr(), part.data_ptr(), part.numel(),
                                 unfed, scratch.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.bn_status_string(st)
    return dx, dw, scratch


@pytest.mark.parametrize("d", [2048, 320, 1024, 2056, 3072, 4096, 4104, 5120, 5128])
def test_norm_backward_matches_oracle(lib, d):
    x, w, dres, rstd, dnp, dx_ref, dw_ref = case(1000, d, seed=d)
    dx, dw, scratch = launch(lib, x, w, dres, rstd, dnp)
    status = lib.bn_get_device_status(ctypes.c_void_p(scratch.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 0
    tol = C.TOL["bf16"]
    e_dx = C.rel_err(dx.float().cpu().numpy().astype(np.float64), dx_ref)
    e_dw = C.rel_err(dw.float().cpu().numpy().astype(np.float64), dw_ref)
    print(f"d={d}: dx {e_dx:.2e}, dw {e_dw:.2e}")
    assert e_dx < tol and e_dw < tol


@pytest.mark.parametrize("d", [2048, 4096, 5120])
def test_unfed_norm_backward_times_out_and_context_survives(lib, d):
    x, w, dres, rstd, dnp, dx_ref, dw_ref = case(1000, d, seed=7)
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    _, _, scratch = launch(lib, x, w, dres, rstd, dnp, unfed=1)
    status = lib.bn_get_device_status(ctypes.c_void_p(scratch.data_ptr()),
                                      ctypes.c_void_p(stream.cuda_stream))
    waited = time.perf_counter() - t0
    assert status == 5, lib.bn_status_string(status)      # BN_ERR_TIMEOUT
    assert 0.5 < waited < 30.0                             # the 1 s limit, not a hang
    # the context is intact: the same launch, fed
    dx, dw, scratch = launch(lib, x, w, dres, rstd, dnp)
    assert lib.bn_get_device_status(ctypes.c_void_p(scratch.data_ptr()),
                                    ctypes.c_void_p(stream.cuda_stream)) == 0
    assert C.rel_err(dx.float().cpu().numpy().astype(np.float64), dx_ref) < C.TOL["bf16"]
    assert C.rel_err(dw.float().cpu().numpy().astype(np.float64), dw_ref) < C.TOL["bf16"]
