"""CPU tests of the C ABI: the library builds, loads, exports every declared
symbol, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from weight_streaming_expert_gb300 import build_lib, native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    names = re.findall(r"\b(moe_[a-z_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return native.lib()


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ("moe_create", "moe_forward", "moe_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 10
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, f"not exported: {missing}"


def test_built_for_sm103a_only():
    assert "arch=compute_103a,code=sm_103a" in build_lib.ARCH
    assert os.path.exists(build_lib.LIB)


@pytest.mark.parametrize("args,frag", [
    ((255, 512, 8, 512), "hidden"),
    ((2560 + 256, 512, 8, 512), "hidden"),   # 11 x 256: no kernel instantiation
    ((2560, 512, 8, 384), "inter"),
    ((256, 16, 2, 512), "inter"),            # inter not dividing hidden
    ((1280, 40, 2, 512), "inter"),
    ((2560, 512, 0, 512), "topk"),
    ((2560, 512, 33, 512), "topk"),
    ((2560, 4, 8, 512), "n_experts"),
    ((2560, 2048, 8, 512), "n_experts"),
])
def test_create_rejects_bad_sizes(L, args, frag):
    dummy = ctypes.c_void_p(16)
    h = L.moe_create(*args, dummy, dummy, dummy)
    assert not h
    assert frag in native.last_error()


def test_create_rejects_null_weights(L):
    h = L.moe_create(2560, 512, 8, 512, None, None, None)
    assert not h
    assert "null" in native.last_error()


def test_forward_rejects_null_handle(L):
    assert L.moe_forward(None, None, None, None, 1, None) == native.MOE_ERR_INVALID_ARG
    assert L.moe_forward_ex(None, None, None, None, None, 1, None, 0) == native.MOE_ERR_INVALID_ARG
    assert L.moe_get_status(None) == native.MOE_ERR_INVALID_ARG
    assert L.moe_get_info(None, None) == native.MOE_ERR_INVALID_ARG
    assert L.moe_set_router_bias(None, None) == native.MOE_ERR_INVALID_ARG
    L.moe_destroy(None)  # no-op
    assert "null" in native.last_error()


def test_no_gpu_create_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    dummy = ctypes.c_void_p(16)
    h = L.moe_create(256, 16, 2, 128, dummy, dummy, dummy)
    assert not h
    assert native.last_error()
