"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function declared in include/moe_ffn.h, sizes its buffers by the same
closed form as the oracle, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import CONFIGS
from oracle import routing

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(moe.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe_ffn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[a-z_ ]+[ *]+(\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 14, names
    L = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert set(moe.EXPORTS) == set(names)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_m_sum_bound_matches_oracle(name):
    c = CONFIGS[name]
    for A in (16, 32, 64, 128):
        p = moe.Problem.from_config(c, block_size=A)
        assert moe.moe_m_sum_bound(p) == routing.m_sum_bound(c.M, c.topk, c.E, A)


def test_workspace_sizes_positive_and_monotone():
    p = moe.Problem.from_config(CONFIGS["mixtral"])
    ws = moe.moe_workspace_bytes(p)
    cap = moe.moe_m_sum_bound(p)
    # at least x_perm (shared with y2) + z, both bf16
    assert ws >= cap * p.H * 2 + cap * p.I * 2
    assert moe.moe_host_workspace_bytes(p) > ws
    assert moe.moe_align_workspace_bytes(p) > 0


@pytest.mark.parametrize("bad", [dict(M=-1), dict(M=16385), dict(H=100), dict(I=0), dict(E=0),
                                 dict(E=1025), dict(topk=0), dict(topk=17), dict(block_size=48),
                                 dict(quant="bf16", apply_router_weight_on_input=True)])
def test_invalid_problems_rejected(bad):
    kw = dict(M=16, H=256, I=128, E=8, topk=2)
    kw.update(bad)
    p = moe.Problem(**kw)
    assert moe.moe_m_sum_bound(p) == 0 and moe.moe_workspace_bytes(p) == 0
    L = moe.lib()
    st = L.fused_experts(ctypes.byref(p.c()), *([None] * 9), 0, None)
    assert st == 1  # MOE_ERR_INVALID_ARG, nothing launched


def test_empty_batch_is_a_noop():
    p = moe.Problem(M=0, H=256, I=128, E=8, topk=2)
    L = moe.lib()
    assert L.fused_experts(ctypes.byref(p.c()), *([None] * 9), 0, None) == 0
    assert L.unpermute_reduce(ctypes.byref(p.c()), None, None, None, None, None) == 0


def test_null_pointers_and_small_workspace_rejected():
    p = moe.Problem(M=16, H=256, I=128, E=8, topk=2)
    L = moe.lib()
    dummy = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    args = [dummy] * 9
    st = L.fused_experts(ctypes.byref(p.c()), *args, 1, None)
    assert st == 5  # MOE_ERR_WORKSPACE_TOO_SMALL
    args[0] = None
    assert L.fused_experts(ctypes.byref(p.c()), *args, 1 << 40, None) == 1


@pytest.mark.parametrize("bs", [0, 8, 48, 96, 256])
def test_gemm_block_size_outside_the_validated_set_is_rejected(bs):
    """block_size is one of 16, 32, 64, 128 (the GEMMs cut 128-row tiles
    inside each expert's segment, so every one of them is served); anything
    else is an invalid problem, refused before any launch."""
    p = moe.Problem(M=16, H=256, I=128, E=8, topk=2, block_size=bs)
    L = moe.lib()
    d = ctypes.c_void_p(16)
    assert L.grouped_gemm_w13(ctypes.byref(p.c()), d, None, d, None, d, d, d, None, 1, None) == 1
    assert moe.moe_m_sum_bound(p) == 0


def test_batched_layout_takes_block_size_128_only():
    """The batched layout's blocks are the 128-row tiles themselves."""
    p = moe.Problem(M=16, H=256, I=128, E=8, topk=2, block_size=64)
    assert moe.moe_m_sum_bound(p) > 0
    assert moe.lib().moe_batched_workspace_bytes(ctypes.byref(p.c()), 128) == 0


@pytest.mark.parametrize("M,E,k,scoring", [(-1, 8, 2, 0), (16385, 8, 2, 0), (4, 0, 1, 0),
                                            (4, 1025, 2, 0), (4, 8, 0, 0), (4, 8, 9, 0),
                                            (4, 64, 17, 0), (4, 8, 2, 2)])
def test_router_invalid_arguments_rejected(M, E, k, scoring):
    L = moe.lib()
    dummy = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    st = L.moe_topk_router(M, E, k, dummy, 0, scoring, 1, None, dummy, dummy, None, None)
    assert st == 1   # MOE_ERR_INVALID_ARG


def test_router_empty_batch_and_null_outputs():
    L = moe.lib()
    assert L.moe_topk_router(0, 8, 2, None, 0, 0, 1, None, None, None, None, None) == 0
    dummy = ctypes.c_void_p(16)
    assert L.moe_topk_router(4, 8, 2, dummy, 0, 0, 1, None, None, dummy, None, None) == 1
    assert L.moe_topk_router(4, 8, 2, None, 0, 0, 1, None, dummy, dummy, None, None) == 1


def test_status_strings():
    for code, name in moe.STATUS.items():
        assert moe.moe_status_string(code) == name


def test_gemm2_split_sizes_and_argument_checks():
    """Sizing of the K-sliced GEMM2 and the checks made before any launch
    (no GPU needed: invalid calls return before touching the device)."""
    p = moe.Problem.from_config(CONFIGS["decode"])
    R = p.M * p.topk
    assert moe.moe_gemm2_partial_bytes(p, 7) == 7 * R * p.H * 4
    assert moe.moe_gemm2_partial_bytes(p, 0) == 0
    bad = moe.Problem(M=16, H=100, I=128, E=8, topk=2)
    assert moe.moe_gemm2_splits(bad) == 0 and moe.moe_gemm2_partial_bytes(bad, 2) == 0
    # any valid problem gets a count in [1, 8]; quantised modes never slice
    assert 1 <= moe.moe_gemm2_splits(p) <= 8
    assert moe.moe_gemm2_splits(moe.Problem.from_config(CONFIGS["dsfp8"])) == 1
    L = moe.lib()
    c = ctypes.byref(p.c())
    # null pointers, a slice count above the K steps, a quantised problem
    assert L.grouped_gemm_w2_split(c, None, None, None, None, None, 2, None, None) == 1
    fake = ctypes.c_void_p(0x1000)
    assert L.grouped_gemm_w2_split(c, fake, fake, fake, fake, fake, p.I // 64 + 1, fake,
                                   None) == 1
    q = ctypes.byref(moe.Problem.from_config(CONFIGS["dsfp8"]).c())
    assert L.grouped_gemm_w2_split(q, fake, fake, fake, fake, fake, 2, fake, None) == 1
    # the sliced reduce takes no router weight on the input or in GEMM2
    w = ctypes.byref(moe.Problem(M=16, H=256, I=128, E=8, topk=1,
                                 apply_router_weight_on_input=True).c())
    assert L.unpermute_reduce_split(w, fake, 2, fake, fake, fake, None) == 1
    assert L.unpermute_reduce_split(c, None, 2, None, None, None, None) == 1


def test_align_permute_launch_count():
    """Kernels stage 1 launches (the bench's launch accounting): one-CTA routing
    for small batches (up to 2048 routed items, or 8192 over at most 64 experts),
    else histograms + scan + scatter; plus the permute."""
    want = {"tiny": 2, "mixtral": 2, "decode": 2, "dsfp8": 4, "mxfp4": 4, "mxfp8": 4}
    for name, n in want.items():
        assert moe.moe_align_permute_launches(moe.Problem.from_config(CONFIGS[name])) == n, name
    edge = [(2048, 1, 256, 2), (2049, 1, 256, 4), (4096, 2, 64, 2), (4096, 2, 65, 4),
            (8193, 1, 8, 4)]
    for M, k, E, n in edge:
        assert moe.moe_align_permute_launches(moe.Problem(M=M, H=256, I=128, E=E, topk=k)) == n
    assert moe.moe_align_permute_launches(moe.Problem(M=0, H=256, I=128, E=8, topk=2)) == 0
    assert moe.moe_align_permute_launches(moe.Problem(M=16, H=100, I=128, E=8, topk=2)) == 0
