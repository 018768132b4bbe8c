"""The C-ABI library loads, exports every declared entry point, and its host-side
logic (validation, capacity, sizing) behaves; no device work is done here."""
import ctypes
import os
import re

import pytest

import mixture_experts_ffn_19_b300 as moe
from mixture_experts_ffn_19_b300 import build as moe_build
import oracle
import synth
from helpers import config_of

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "moe_forward" in names and "moe_route" in names and len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_validation(lib):
    good = config_of(synth.WORKLOADS["mixtral_prefill"])
    assert moe.moe_validate_config(good) == moe.MOE_OK
    for field, bad, want in [("n_experts", 0, moe.MOE_ERR_INVALID_ARG),
                             ("n_experts", 257, moe.MOE_ERR_INVALID_ARG),
                             ("top_k", 9, moe.MOE_ERR_INVALID_ARG),
                             ("top_k", 0, moe.MOE_ERR_INVALID_ARG),
                             ("d_model", 4100, moe.MOE_ERR_INVALID_ARG),
                             ("d_ff", 12, moe.MOE_ERR_INVALID_ARG),
                             # MOE_MAX_DIM = 65536 bounds d and F
                             ("d_model", 65536 + 8, moe.MOE_ERR_INVALID_ARG),
                             ("d_ff", 65536 + 8, moe.MOE_ERR_INVALID_ARG),
                             ("d_model", 65536, moe.MOE_OK),
                             ("d_ff", 65536, moe.MOE_OK),
                             ("n_tokens", -1, moe.MOE_ERR_INVALID_ARG),
                             ("cap_mode", 3, moe.MOE_ERR_INVALID_ARG),
                             ("alpha", 0.0, moe.MOE_ERR_INVALID_ARG),
                             ("bias_mode", 2, moe.MOE_ERR_INVALID_ARG),
                             ("bias_mode", -1, moe.MOE_ERR_INVALID_ARG),
                             ("act", moe.MOE_ACT_GELU, moe.MOE_ERR_UNSUPPORTED)]:
        c = config_of(synth.WORKLOADS["mixtral_prefill"])
        setattr(c, field, bad)
        assert moe.moe_validate_config(c) == want, field
    small = config_of(synth.WORKLOADS["tiny_fp32"])
    small.top_k = 9
    assert moe.moe_validate_config(small) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_workspace_size(small) == 0


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_capacity_matches_oracle(lib, name):
    w = synth.WORKLOADS[name]
    c = config_of(w)
    want = oracle.capacity(w.n_tokens, w.n_experts, w.top_k, w.alpha) if w.cap_mode else -1
    assert moe.moe_capacity(c) == want
    # the worked example of the capacity section: N=32, E=64, k=2, alpha=1.2 -> 1
    c2 = moe.make_config(32, 64, 64, 2, 64, cap_mode=moe.MOE_CAP_DROP, alpha=1.2)
    assert moe.moe_capacity(c2) == 1


@pytest.mark.parametrize("alpha", [0.7, 0.3, 0.6, 1.1, 1.3, 0.9, 2.2, 1.25, 4.0])
def test_capacity_factor_is_taken_exactly(lib, alpha):
    # factors with no exact binary form, where floor(k N / E) * alpha is an
    # integer: 1250 * 0.7 = 875, 1000 * 0.3 = 300, ...  A single-precision
    # factor (0.7 -> 0.69999999) would floor one lower than the oracle
    for n, e, k in [(40000, 64, 2), (16000, 32, 2), (5000, 10, 2), (100, 10, 1), (6400, 64, 8)]:
        c = moe.make_config(n, 64, e, k, 64, cap_mode=moe.MOE_CAP_REROUTE, alpha=alpha)
        assert moe.moe_capacity(c) == oracle.capacity(n, e, k, alpha), (n, e, k, alpha)
    c = moe.make_config(40000, 64, 64, 2, 64, cap_mode=moe.MOE_CAP_DROP, alpha=0.7)
    assert moe.moe_capacity(c) == 875


def test_sizes(lib):
    w = synth.WORKLOADS["dsv2"]
    c = config_of(w)
    assert moe.moe_max_rows(c) == w.n_tokens * w.top_k + w.n_experts * 127
    assert moe.moe_max_total_rows(c) == moe.moe_max_rows(c) + 2 * 8192
    assert moe.moe_workspace_size(c) % 256 == 0
    assert moe.moe_workspace_size(c) > moe.moe_max_total_rows(c) * w.d_model * 2


def test_null_arguments_are_rejected_before_any_launch(lib):
    c = config_of(synth.WORKLOADS["tiny_fp32"])
    st = lib.moe_route(ctypes.byref(c), None, None, None, None, None, None, None, None, 0, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = lib.moe_forward(ctypes.byref(c), None, None, None, None, None, None, None, None, None,
                         None, None, 0, None, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = lib.moe_combine(ctypes.byref(c), None, None, None, None, None, None, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert moe.status_string(moe.MOE_ERR_WORKSPACE) == "workspace too small"


def test_zero_tokens_and_tiny_shapes_size_without_error(lib):
    for n in (0, 1, 127, 129):
        c = moe.make_config(n, 64, 4, 2, 64, n_shared=1, cap_mode=moe.MOE_CAP_REROUTE, alpha=1.0)
        assert moe.moe_validate_config(c) == moe.MOE_OK
        assert moe.moe_workspace_size(c) > 0
    c = moe.make_config(0, 128, 8, 2, 256, act=moe.MOE_ACT_GELU, dtype=moe.MOE_F32, has_ffn_bias=True)
    assert moe.moe_workspace_size(c) > 0


def test_selftest_rejects_missing_workspace(lib):
    # host-side checks only: nothing is launched
    assert lib.moe_selftest_timeout(None, 0, 1000, None) == moe.MOE_ERR_INVALID_ARG


def test_fp8_ffn_refuses_the_workspace_x_perm(lib):
    # the E4M3 expert FFN writes f16 copies of the token rows into the
    # workspace's own x_perm, so that buffer cannot also be the input; the
    # check is made before any launch (fake device addresses, nothing is read)
    c = moe.make_config(32, 256, 8, 2, 512)
    n = moe.moe_workspace_size(c)
    ws = 1 << 36
    v = moe.moe_views()
    assert lib.moe_workspace_views(ctypes.byref(c), ws, n, ctypes.byref(v)) == moe.MOE_OK
    fake = 1 << 40
    st = lib.moe_expert_ffn_fp8(ctypes.byref(c), fake, v.x_perm, fake, fake, fake, fake, fake,
                                fake, fake, ws, n, None)
    assert st == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("n,e,k,s", [(1, 1, 1, 1), (32, 160, 6, 2), (64, 8, 2, 1), (127, 4, 4, 3),
                                      (300, 64, 2, 1), (4097, 256, 8, 8)])
def test_shared_f16_copy_fits_past_the_routed_rows(lib, n, e, k, s):
    # with E4M3 weights the shared experts read an f16 copy of x placed in
    # y_perm after the routed region: rows [max_rows, max_rows + N) must exist
    c = moe.make_config(n, 64, e, k, 64, n_shared=s)
    assert moe.moe_max_total_rows(c) >= moe.moe_max_rows(c) + n
    # and the routed rows a dispatch can produce stay inside max_rows
    assert moe.moe_max_rows(c) >= n * k + e * 127
