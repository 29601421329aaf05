"""Unit tests of the GEMM engine behind the block (tensor-core bf16 and FFMA fp32):
every fused epilogue, every operand layout the block uses, ragged and tiny
shapes, K split of left-over tiles, grouped launches. Reference: the same op in numpy float64 on
the exact (bf16-rounded) inputs. Padding around every operand and output holds
NaN, so any read or write outside the logical bounds fails the test."""
import zlib

import numpy as np
import pytest

from rank_bottleneck_gb300.synth import round_to_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f32": 1e-5}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_bottleneck_gb300 import _build
    _build.build()
    from rank_bottleneck_gb300 import block as B
    return B.load()


def tdt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def rnd(rng, shape, dtype, scale=1.0):
    a = (rng.standard_normal(shape) * scale).astype(np.float32)
    return round_to_bf16(a) if dtype == "bf16" else a


def operand(L, mn_major, dtype):
    """Store logical [MN, K] as [MN, ld>=K] or [K, ld>=MN]; padding = NaN."""
    S = L.T if mn_major else L
    rows, cols = S.shape
    ld = (cols + 7) // 8 * 8 + 8
    buf = np.full((rows, ld), np.nan, dtype=np.float32)
    buf[:, :cols] = S
    return torch.from_numpy(buf).to("cuda", tdt(dtype)), ld


def out_buf(M, N, dtype):
    ld = (N + 7) // 8 * 8 + 8
    return torch.full((M, ld), float("nan"), dtype=tdt(dtype), device="cuda"), ld


def host(t, N):
    a = t.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isnan(a[:, N:])), "wrote outside the output columns"
    return a[:, :N]


def in_buf(A, dtype, ld):
    buf = np.full((A.shape[0], ld), np.nan, dtype=np.float32)
    buf[:, :A.shape[1]] = A
    return torch.from_numpy(buf).to("cuda", tdt(dtype))


def err(got, ref):
    return np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30)


def silu(z):
    return z / (1 + np.exp(-z))


def dsilu(z):
    s = 1 / (1 + np.exp(-z))
    return s * (1 + z * (1 - s))


def problem(rng, M, N, K, a_mn, b_mn, dtype, two=False):
    A = rnd(rng, (M, K), dtype)
    Bm = rnd(rng, (N, K), dtype, 1 / np.sqrt(K))
    ta, lda = operand(A, a_mn, dtype)
    tb, ldb = operand(Bm, b_mn, dtype)
    q = dict(M=M, N=N, K=K, a=ta, b=tb, lda=lda, ldb=ldb, a_mn=a_mn, b_mn=b_mn)
    ref = dict(A=A.astype(np.float64), B=Bm.astype(np.float64))
    if two:
        A2 = rnd(rng, (M, K), dtype)
        B2 = rnd(rng, (N, K), dtype, 1 / np.sqrt(K))
        ta2, lda2 = operand(A2, a_mn, dtype)
        tb2, ldb2 = operand(B2, b_mn, dtype)
        assert lda2 == lda and ldb2 == ldb
        q.update(a2=ta2, b2=tb2)
        ref.update(A2=A2.astype(np.float64), B2=B2.astype(np.float64))
    return q, ref


LAYOUTS = [(False, False), (False, True), (True, True)]
SHAPES = [(128, 256, 64), (300, 520, 200), (1000, 384, 1024), (77, 40, 24), (1, 8, 8),
          (130, 333, 205), (67, 5, 3)]  # ragged N and K (not multiples of 8)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: f"a{'MN' if l[0] else 'K'}-b{'MN' if l[1] else 'K'}")
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_store(lib, dtype, layout, shape):
    from _gemmhook import run
    rng = np.random.default_rng(zlib.crc32(repr((dtype, layout, shape)).encode()))
    M, N, K = shape
    q, r = problem(rng, M, N, K, *layout, dtype)
    q["out0"], q["ldo"] = out_buf(M, N, dtype)
    run(lib, "store", [q], dtype=dtype)
    assert err(host(q["out0"], N), r["A"] @ r["B"].T) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_store_split_k_with_row_and_column_scales(lib, dtype):
    from _gemmhook import run
    rng = np.random.default_rng(7)
    M, N, K = 256, 520, 8192 if dtype == "bf16" else 1024
    q, r = problem(rng, M, N, K, True, True, dtype)
    colv = rnd(rng, (N,), dtype) + 1
    q["colv"] = torch.from_numpy(colv).to("cuda", tdt(dtype))
    q["out0"], q["ldo"] = out_buf(M, N, dtype)
    run(lib, "store", [q], dtype=dtype, allow_split=True)
    ref = (r["A"] @ r["B"].T) * colv.astype(np.float64)[None]
    assert err(host(q["out0"], N), ref) <= TOL[dtype]
    # the same with a row scale (never split)
    q2, r2 = problem(rng, 200, 136, 96, False, True, dtype)
    rowv = (rng.random(200) + 0.5).astype(np.float32)
    q2["rowv"] = torch.from_numpy(rowv).cuda()
    q2["out0"], q2["ldo"] = out_buf(200, 136, dtype)
    run(lib, "store", [q2], dtype=dtype, allow_split=True)
    ref2 = (r2["A"] @ r2["B"].T) * rowv.astype(np.float64)[:, None]
    assert err(host(q2["out0"], 136), ref2) <= TOL[dtype]


# K split of the tiles left over after whole rounds of CTA groups (76 pairs on a
# 152-SM GB300): fewer tiles than groups (all split), more tiles with a
# remainder, an exact multiple (no split), and a launch of many problems like
# the block's gathered weight gradients (ragged shapes, with and without a
# column scale).
SPLIT_CASES = {
    "fewer-tiles": [(1536, 2048, 16384)],
    "remainder": [(2816, 2048, 8192)],
    "exact-rounds": [(4864, 1024, 4096)],
    "eleven-problems": [(512, 5464, 4096), (520, 264, 4096), (2048, 512, 4096), (512, 2048, 4096),
                        (5461, 512, 4096), (5461, 512, 4096), (1024, 2048, 4096), (2048, 512, 4096),
                        (2048, 512, 4096), (2048, 512, 4096), (512, 2048, 4096)],
}


@pytest.mark.parametrize("case", list(SPLIT_CASES))
def test_store_split_remainder(lib, case):
    from _gemmhook import run
    rng = np.random.default_rng(zlib.crc32(case.encode()))
    qs, refs = [], []
    for i, (M, N, K) in enumerate(SPLIT_CASES[case]):
        q, r = problem(rng, M, N, K, True, True, "bf16")
        ref = r["A"] @ r["B"].T
        if i % 2:
            colv = rnd(rng, (N,), "bf16") + 1
            q["colv"] = torch.from_numpy(colv).to("cuda", torch.bfloat16)
            ref = ref * colv.astype(np.float64)[None]
        q["out0"], q["ldo"] = out_buf(M, N, "bf16")
        qs.append(q)
        refs.append(ref)
    run(lib, "store", qs, dtype="bf16", allow_split=True)
    for q, ref, (M, N, K) in zip(qs, refs, SPLIT_CASES[case]):
        assert err(host(q["out0"], N), ref) <= TOL["bf16"]


def test_split_k_is_deterministic(lib):
    from _gemmhook import run
    rng = np.random.default_rng(8)
    q, _ = problem(rng, 2816, 2048, 8192, True, True, "bf16")  # whole rounds + split tiles
    outs = []
    for _ in range(2):
        q["out0"], q["ldo"] = out_buf(2816, 2048, "bf16")
        run(lib, "store", [q], dtype="bf16", allow_split=True)
        outs.append(q["out0"][:, :2048].clone())
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("sigma", [0, 1])
def test_sigma(lib, dtype, sigma):
    from _gemmhook import run
    rng = np.random.default_rng(9)
    M, N, K = 333, 264, 192
    q, r = problem(rng, M, N, K, False, False, dtype)
    q["out0"], q["ldo"] = out_buf(M, N, dtype)
    q["out1"], _ = out_buf(M, N, dtype)
    run(lib, "sigma", [q], dtype=dtype, sigma=sigma)
    z = r["A"] @ r["B"].T
    assert err(host(q["out0"], N), z) <= TOL[dtype]
    assert err(host(q["out1"], N), silu(z) if sigma else z) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("S", [1, 2, 4, 8])
def test_online_norm(lib, dtype, S):
    from _gemmhook import run
    rng = np.random.default_rng(10 + S)
    M, N, K, eps = 260, 200, 512, 1e-5
    q, r = problem(rng, M, N, K, False, False, dtype)
    A = r["A"].copy()
    A[3, : K // S] = 0.0  # a zero shard in one row
    q["a"], _ = operand(A.astype(np.float32), False, dtype)
    ss = np.stack([np.sum(A[:, s * K // S:(s + 1) * K // S] ** 2, axis=1) for s in range(S)], 1)
    q["rowv"] = torch.from_numpy(ss.astype(np.float32)).cuda()
    q["out0"], q["ldo"] = out_buf(M, N, dtype)
    q["out1"], _ = out_buf(M, N, dtype)
    run(lib, "norm", [q], dtype=dtype, S=S, eps=eps)
    rms = np.sqrt(np.sum(ss, 1) / K + eps)
    z = (A @ r["B"].T) / rms[:, None]
    assert err(host(q["out0"], N), z) <= TOL[dtype]
    assert err(host(q["out1"], N), silu(z)) <= TOL[dtype]


@pytest.mark.parametrize("S", [4, 8])
def test_online_norm_many_tiles(lib, S):
    """More 256-row tiles than CTA pairs, with a ragged last tile: every pair runs
    several tiles, so each shard's partial product cycles through the TMEM slot
    ring across tile boundaries."""
    from _gemmhook import run
    rng = np.random.default_rng(40 + S)
    M, N, K, eps = 5156, 1024, 1024, 1e-5
    q, r = problem(rng, M, N, K, False, False, "bf16")
    A = r["A"]
    ss = np.stack([np.sum(A[:, s * K // S:(s + 1) * K // S] ** 2, axis=1) for s in range(S)], 1)
    q["rowv"] = torch.from_numpy(ss.astype(np.float32)).cuda()
    q["out0"], q["ldo"] = out_buf(M, N, "bf16")
    q["out1"], _ = out_buf(M, N, "bf16")
    run(lib, "norm", [q], dtype="bf16", S=S, eps=eps)
    rms = np.sqrt(np.sum(ss, 1) / K + eps)
    z = (A @ r["B"].T) / rms[:, None]
    assert err(host(q["out0"], N), z) <= TOL["bf16"]
    assert err(host(q["out1"], N), silu(z)) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_resid_and_grouped(lib, dtype):
    from _gemmhook import run
    rng = np.random.default_rng(11)
    probs, refs = [], []
    for N in (256, 128, 203):
        q, r = problem(rng, 500, N, 128, False, False, dtype)
        R = rnd(rng, (500, N), dtype)
        q["out0"], q["ldo"] = out_buf(500, N, dtype)
        q["in0"] = in_buf(R, dtype, q["ldo"])
        q["ldi"] = q["ldo"]
        probs.append(q)
        refs.append(R + r["A"] @ r["B"].T)
    run(lib, "resid", probs, dtype=dtype)
    for q, ref in zip(probs, refs):
        assert err(host(q["out0"], q["N"]), ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_swiglu(lib, dtype):
    from _gemmhook import run
    rng = np.random.default_rng(12)
    M, N, K = 300, 333, 128
    q, r = problem(rng, M, N, K, False, False, dtype, two=True)
    q["out0"], q["ldo"] = out_buf(M, N, dtype)
    q["out1"], _ = out_buf(M, N, dtype)
    q["out2"], _ = out_buf(M, N, dtype)
    run(lib, "swiglu", [q], dtype=dtype)
    G = r["A"] @ r["B"].T
    U = r["A2"] @ r["B2"].T
    assert err(host(q["out0"], N), G) <= TOL[dtype]
    assert err(host(q["out1"], N), U) <= TOL[dtype]
    assert err(host(q["out2"], N), silu(G) * U) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_dsigma_and_dswiglu(lib, dtype):
    from _gemmhook import run
    rng = np.random.default_rng(13)
    M, N, K = 270, 141, 317
    rowv = (rng.random(M) + 0.5).astype(np.float32)
    q, r = problem(rng, M, N, K, False, True, dtype)
    Z = rnd(rng, (M, N), dtype, 2.0)
    q["out0"], q["ldo"] = out_buf(M, N, dtype)
    q["in0"] = in_buf(Z, dtype, q["ldo"])
    q["ldi"] = q["ldo"]
    q["rowv"] = torch.from_numpy(rowv).cuda()
    run(lib, "dsigma", [q], dtype=dtype, sigma=1)
    acc = r["A"] @ r["B"].T
    assert err(host(q["out0"], N), acc * dsilu(Z) * rowv[:, None]) <= TOL[dtype]

    q, r = problem(rng, M, N, K, False, True, dtype)
    G = rnd(rng, (M, N), dtype, 2.0)
    U = rnd(rng, (M, N), dtype)
    q["out0"], q["ldo"] = out_buf(M, N, dtype)
    q["out1"], _ = out_buf(M, N, dtype)
    q["in0"] = in_buf(G, dtype, q["ldo"])
    q["in1"] = in_buf(U, dtype, q["ldo"])
    q["ldi"] = q["ldo"]
    q["rowv"] = torch.from_numpy(rowv).cuda()
    run(lib, "dswiglu", [q], dtype=dtype)
    dm = r["A"] @ r["B"].T
    assert err(host(q["out0"], N), dm * U * dsilu(G) * rowv[:, None]) <= TOL[dtype]
    assert err(host(q["out1"], N), dm * silu(G) * rowv[:, None]) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chain(lib, dtype):
    from _gemmhook import run
    rng = np.random.default_rng(14)
    M, N, K = 260, 262, 203
    q, r = problem(rng, M, N, K, False, True, dtype, two=True)
    q["out0"], q["ldo"] = out_buf(M, N, dtype)
    run(lib, "chain", [q], dtype=dtype)
    ref = r["A"] @ r["B"].T + r["A2"] @ r["B2"].T
    assert err(host(q["out0"], N), ref) <= TOL[dtype]


@pytest.mark.parametrize("S", [2, 4, 8, 16])
def test_online_norm_fp32_shards_match_one_shard(lib, S):
    """The Online RMSNorm epilogue with S shards equals S = 1 to 1e-6 in fp32."""
    from _gemmhook import run
    rng = np.random.default_rng(20 + S)
    M, N, K = 300, 264, 1024
    q, r = problem(rng, M, N, K, False, False, "f32")
    A = r["A"]
    outs = {}
    for s in (1, S):
        ss = np.stack([np.sum(A[:, j * K // s:(j + 1) * K // s] ** 2, axis=1) for j in range(s)], 1)
        q["rowv"] = torch.from_numpy(ss.astype(np.float32)).cuda()
        q["out0"], q["ldo"] = out_buf(M, N, "f32")
        q["out1"] = None
        run(lib, "norm", [q], dtype="f32", S=s)
        outs[s] = host(q["out0"], N)
    assert err(outs[S], outs[1]) <= 1e-6
