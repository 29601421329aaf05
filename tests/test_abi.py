"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the header declares, sizes workspaces, and rejects bad
arguments synchronously, before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h)
           for h in ("boostblk.h", "boostattn.h", "boostblk_testing.h")]


@pytest.fixture(scope="module")
def lib():
    from rank_bottleneck_gb300 import _build
    _build.build()
    from rank_bottleneck_gb300 import block as B
    return B.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(bn_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert "bn_block_forward" in names and "bn_block_backward" in names
    assert "bn_attn_forward" in names and "bn_attn_backward" in names
    for n in names:
        assert hasattr(lib, n), n


def cfg(**kw):
    from rank_bottleneck_gb300.block import BlockConfig
    base = dict(T=16384, d=2048, r=512, d_ff=5461, S=4)
    base.update(kw)
    return BlockConfig(**base)


def test_workspace_sizes_and_checkpoint_saving():
    from rank_bottleneck_gb300.block import workspace_size
    saved, scratch = workspace_size(cfg())
    saved_ck, scratch_ck = workspace_size(cfg(checkpoint=True))
    T, d, r = 16384, 2048, 512
    # checkpoint mode saves exactly the four pre-activation tensors, [T, 7r] bf16
    assert abs(saved_ck - T * 7 * r * 2) <= 4 * 256
    assert saved > 5 * saved_ck
    assert scratch_ck > scratch  # the recomputed activations live in scratch instead


def test_workspace_with_uneven_ranks():
    """Checkpoint mode saves the pre-activations of every layer: T x sum(r_i)."""
    from rank_bottleneck_gb300.block import workspace_size
    ranks = (384, 384, 768, 256, 640, 640, 512)
    saved_ck, _ = workspace_size(cfg(checkpoint=True, ranks=ranks))
    assert abs(saved_ck - 16384 * sum(ranks) * 2) <= 4 * 256
    # all ranks given explicitly equal to r: the same sizes as the even block
    assert workspace_size(cfg(ranks=(512,) * 7)) == workspace_size(cfg())


@pytest.mark.parametrize("bad, code", [
    (dict(dtype="f32", S=3), 1),          # d % S != 0
    (dict(d_ff=100, ld_ff=50), 1),        # ld_ff < d_ff
    (dict(ld_ff=5462), 2),                # 16-byte rows of d_ff-wide tensors
    (dict(r=500), 2),                     # rank must be a multiple of 8
    (dict(S=17), 1),
    (dict(dense=True, checkpoint=True), 3),
    (dict(S=64), 1),
    (dict(d=512, S=16), 3),               # bf16 shards narrower than 64 columns
    (dict(dense=True, btp=True), 3),      # the TP emulation is of the factorised block
    (dict(d_ff=100, ld_ff=128, d=1024, S=4, btp=True), 3),  # fewer 64-column blocks than shards
    (dict(ranks=(512, 512, 500, 512, 512, 512, 512)), 2),  # a layer's rank not a multiple of 8
    (dict(ranks=(512, -8, 512, 512, 512, 512, 512)), 1),   # a negative rank
    (dict(dense=True, ranks=(8, 0, 0, 0, 0, 0, 0)), 1),    # the dense block has no ranks
])
def test_bad_descriptors_are_rejected(lib, bad, code):
    from rank_bottleneck_gb300.block import workspace_size
    c = cfg(**bad)
    with pytest.raises(RuntimeError) as e:
        workspace_size(c)
    assert ["BN_ERR_INVALID_ARG", "BN_ERR_ALIGNMENT", "BN_ERR_UNSUPPORTED"][code - 1] in str(e.value)


def _params_struct(**ptrs):
    from rank_bottleneck_gb300.block import PARAM_NAMES, _Params
    p = _Params()
    for n in PARAM_NAMES:
        setattr(p, n, ptrs.get(n))
    return p


def test_pointer_checks_before_any_launch(lib):
    from rank_bottleneck_gb300.block import PARAM_NAMES
    c = cfg(T=256, d=256, r=64, d_ff=688, dtype="f32")
    d = c.desc()
    good = {n: 4096 * (i + 1) for i, n in enumerate(PARAM_NAMES)}
    # a misaligned parameter pointer
    bad = dict(good, B_q=good["B_q"] + 4)
    st = lib.bn_block_forward(ctypes.byref(d), ctypes.byref(_params_struct(**bad)), 1 << 20,
                              1 << 21, 1 << 22, 1 << 23, 1 << 24, 1 << 25, None)
    assert lib.bn_status_string(st) == b"BN_ERR_ALIGNMENT"
    # a missing parameter
    miss = dict(good)
    miss.pop("A_o")
    st = lib.bn_block_forward(ctypes.byref(d), ctypes.byref(_params_struct(**miss)), 1 << 20,
                              1 << 21, 1 << 22, 1 << 23, 1 << 24, 1 << 25, None)
    assert lib.bn_status_string(st) == b"BN_ERR_INVALID_ARG"
    # the MLP kind must not get attention-half tensors
    m = cfg(T=256, d=256, r=64, d_ff=688, dtype="f32", kind="mlp").desc()
    st = lib.bn_block_forward(ctypes.byref(m), ctypes.byref(_params_struct(**good)), 1 << 20,
                              1 << 21, None, None, 1 << 24, 1 << 25, None)
    assert lib.bn_status_string(st) == b"BN_ERR_INVALID_ARG"
    # dense blocks take no up-projection factors
    dn = cfg(T=256, d=256, r=64, d_ff=688, dtype="f32", dense=True).desc()
    st = lib.bn_block_forward(ctypes.byref(dn), ctypes.byref(_params_struct(**good)), 1 << 20,
                              1 << 21, 1 << 22, 1 << 23, 1 << 24, 1 << 25, None)
    assert lib.bn_status_string(st) == b"BN_ERR_INVALID_ARG"
    assert lib.bn_last_launch_count() == 0


def test_status_strings(lib):
    for code, name in enumerate([b"BN_OK", b"BN_ERR_INVALID_ARG", b"BN_ERR_ALIGNMENT",
                                 b"BN_ERR_UNSUPPORTED", b"BN_ERR_CUDA", b"BN_ERR_TIMEOUT"]):
        assert lib.bn_status_string(code) == name


# ---------------------------------------------------------------------------
# attention core (include/boostattn.h)
# ---------------------------------------------------------------------------

def test_attention_workspace_sizes(lib):
    from rank_bottleneck_gb300.attention import AttnConfig, workspace_size
    c = AttnConfig(B=4, L=4096, H=16)
    assert c.lse_stride == 4096
    assert AttnConfig(B=1, L=1000, H=2).lse_stride == 1024
    n_lse, n_scratch = workspace_size(c)
    assert n_lse == 4 * 16 * 4096 * 4
    assert n_scratch == 256 + 2 * n_lse


@pytest.mark.parametrize("bad, code", [
    (dict(B=0), 1), (dict(L=0), 1), (dict(H=0), 1), (dict(causal=2), 1),
    (dict(d_head=64), 3),                 # only d_head = 128 is built
])
def test_attention_bad_descriptors(lib, bad, code):
    from rank_bottleneck_gb300 import attention as A
    base = dict(B=2, L=256, H=2, d_head=128, causal=1)
    base.update(bad)
    d = A._AttnDesc(base["B"], base["L"], base["H"], base["d_head"], base["causal"])
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert A._lib().bn_attn_workspace_size(ctypes.byref(d), ctypes.byref(a), ctypes.byref(b)) == code
    fake = [ctypes.c_void_p(4096 * (i + 1)) for i in range(7)]
    assert A._lib().bn_attn_forward(ctypes.byref(d), *fake) == code


def test_attention_bad_pointers_rejected_before_launch(lib):
    from rank_bottleneck_gb300 import attention as A
    d = A.AttnConfig(B=2, L=256, H=2).desc()
    ok = [ctypes.c_void_p(4096 * (i + 1)) for i in range(11)]
    f, bw = A._lib().bn_attn_forward, A._lib().bn_attn_backward
    for i in range(6):                    # q, k, v, o, lse, scratch
        args = list(ok[:7])
        args[i] = None
        assert f(ctypes.byref(d), *args) == 1
        args[i] = ctypes.c_void_p(4096 * 9 + 8)
        assert f(ctypes.byref(d), *args) == 2
    for i in range(10):                   # q, k, v, o, lse, dout, dq, dk, dv, scratch
        args = list(ok[:11])
        args[i] = None
        assert bw(ctypes.byref(d), *args) == 1
        args[i] = ctypes.c_void_p(4096 * 20 + 4)
        assert bw(ctypes.byref(d), *args) == 2


@pytest.mark.parametrize("bad, code", [
    (dict(seq_len=0), 1), (dict(seq_len=100), 1),     # T % seq_len != 0
    (dict(kind="mlp"), 1),                            # the attention core needs the full block
    (dict(dtype="f32"), 3),                           # bf16 only
    (dict(d=192, S=3), 3),                            # heads of 128
])
def test_block_attention_descriptor_checks(lib, bad, code):
    from rank_bottleneck_gb300.block import BlockConfig
    kw = dict(T=256, d=256, r=64, d_ff=333, S=4, attn=True, seq_len=128)
    kw.update(bad)
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.bn_block_workspace_size(ctypes.byref(BlockConfig(**kw).desc()), ctypes.byref(a),
                                       ctypes.byref(b)) == code


def test_block_attention_workspace_holds_q_k_o_and_lse(lib):
    from rank_bottleneck_gb300.block import BlockConfig, workspace_size
    base = dict(T=16384, d=2048, r=512, d_ff=5461, S=4)
    s0, c0 = workspace_size(BlockConfig(**base))
    s1, c1 = workspace_size(BlockConfig(**base, attn=True, seq_len=4096))
    T, d = 16384, 2048
    lse = 4 * 16 * 4096 * 4
    assert abs((s1 - s0) - (3 * T * d * 2 + lse)) <= 4 * 256
    assert c1 - c0 >= 3 * T * d * 2 + 2 * lse


def test_attention_flop_model():
    """Visible (query, key) pairs of the causal core: L (L + 1) / 2 per sequence
    and head; the model counts 12 x 128 FLOPs per pair (forward q.k and p v,
    backward dv, dp, dq, dk), the hardware 6 x 128 more (the backward's
    recomputed q.k twice and do.v once)."""
    from rank_bottleneck_gb300.block import BlockConfig
    from rank_bottleneck_gb300.configs import WORKLOADS, attn_pairs, model_flops, recompute_flops
    base = BlockConfig(**WORKLOADS["1b-T16384-d2048-r512-dff5461"])
    layer = BlockConfig(**WORKLOADS["1b-attn-T16384-L4096-d2048-r512-dff5461"])
    pairs = 4 * 16 * 4096 * 4097 / 2
    assert attn_pairs(layer) == pairs and attn_pairs(base) == 0
    assert model_flops(layer) - model_flops(base) == 12 * 128 * pairs
    assert recompute_flops(layer) == 6 * 128 * pairs


def test_attention_unfed_hook_rejects_bad_arguments(lib):
    from rank_bottleneck_gb300 import attention as A
    fn = lib.bn_testing_attn_forward_unfed
    fn.argtypes = [ctypes.POINTER(A._AttnDesc)] + [ctypes.c_void_p] * 7
    fn.restype = ctypes.c_int
    d = A.AttnConfig(B=1, L=128, H=1, d_head=64).desc()
    fake = [ctypes.c_void_p(4096 * (i + 1)) for i in range(7)]
    assert fn(ctypes.byref(d), *fake) == 3                     # d_head 64: unsupported
    d = A.AttnConfig(B=1, L=128, H=1).desc()
    args = list(fake)
    args[0] = None
    assert fn(ctypes.byref(d), *args) == 1                     # q missing
