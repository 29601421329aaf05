"""ctypes binding of bn_testing_gemm (include/boostblk_testing.h) for engine unit tests."""
import ctypes

import torch

EPI = dict(store=0, sigma=1, norm=2, resid=3, swiglu=4, dsigma=5, dswiglu=6, chain=7)


class Problem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("a", ctypes.c_void_p), ("a2", ctypes.c_void_p), ("lda", ctypes.c_int64),
                ("a_mn_major", ctypes.c_int32),
                ("b", ctypes.c_void_p), ("b2", ctypes.c_void_p), ("ldb", ctypes.c_int64),
                ("b_mn_major", ctypes.c_int32),
                ("out0", ctypes.c_void_p), ("out1", ctypes.c_void_p), ("out2", ctypes.c_void_p),
                ("ldo", ctypes.c_int64),
                ("in0", ctypes.c_void_p), ("in1", ctypes.c_void_p), ("ldi", ctypes.c_int64),
                ("rowv", ctypes.c_void_p), ("colv", ctypes.c_void_p)]


def _p(t):
    return None if t is None else t.data_ptr()


def run(lib, epi, probs, *, dtype, sigma=1, S=1, eps=1e-5, allow_split=False,
        scratch_bytes=256 << 20):
    """probs: list of dicts with tensors a, b (a2, b2), out0.. and sizes M, N, K."""
    fn = lib.bn_testing_gemm
    fn.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_float, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.POINTER(Problem), ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    arr = (Problem * len(probs))()
    for i, q in enumerate(probs):
        arr[i] = Problem(q["M"], q["N"], q["K"], _p(q["a"]), _p(q.get("a2")), q["lda"],
                         int(q.get("a_mn", False)), _p(q["b"]), _p(q.get("b2")), q["ldb"],
                         int(q.get("b_mn", False)), _p(q.get("out0")), _p(q.get("out1")),
                         _p(q.get("out2")), q.get("ldo", q["N"]), _p(q.get("in0")),
                         _p(q.get("in1")), q.get("ldi", q["N"]), _p(q.get("rowv")),
                         _p(q.get("colv")))
    scratch = torch.zeros(scratch_bytes, dtype=torch.uint8, device="cuda")
    st = fn(1 if dtype == "bf16" else 0, EPI[epi], sigma, S, eps, int(allow_split), len(probs),
            arr, scratch.data_ptr(), scratch_bytes, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, lib.bn_status_string(st)
    status = int(scratch[:4].view(torch.int32).item())
    assert status == 0, f"device status {status}"
