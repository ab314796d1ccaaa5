"""CPU tests of the C ABI: the library builds, loads, exports every declared
symbol, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from weight_streaming_expert_gb300 import build_lib, native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    src = "\n".join(open(h).read() for h in HEADERS)
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
    for n in ("moe_create", "moe_forward", "moe_destroy",
              "moe_lm_head_create", "moe_lm_head_forward", "moe_lm_head_destroy"):
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


@pytest.mark.parametrize("hidden,vocab,frag", [(255, 1000, "hidden"), (2816, 1000, "hidden"),
                                               (2560, 0, "vocab"), (2560, (1 << 24) + 1, "vocab")])
def test_lm_head_create_rejects_bad_sizes(L, hidden, vocab, frag):
    assert not L.moe_lm_head_create(hidden, vocab, ctypes.c_void_p(16))
    assert frag in native.last_error()


def test_lm_head_rejects_null_and_misaligned_weights(L):
    assert not L.moe_lm_head_create(2560, 1000, None)
    assert not L.moe_lm_head_create(2560, 1000, ctypes.c_void_p(24))
    assert "aligned" in native.last_error()


def test_lm_head_forward_rejects_null_handle(L):
    assert L.moe_lm_head_forward(None, None, None, 1, None) == native.MOE_ERR_INVALID_ARG
    assert L.moe_lm_head_get_status(None) == native.MOE_ERR_INVALID_ARG
    L.moe_lm_head_destroy(None)  # no-op


@pytest.mark.parametrize("rows,k,M,engine,status,frag", [
    (12, 256, 1, 0, native.MOE_ERR_INVALID_ARG, "rows"),    # rows not a multiple of 8
    (16, 288, 1, 0, native.MOE_ERR_INVALID_ARG, "k ="),     # k not a multiple of 256
    (16, 3328, 1, 1, native.MOE_ERR_INVALID_ARG, "k ="),    # k above 3072
    (16, 256, 1, 5, native.MOE_ERR_INVALID_ARG, "engine"),
    (16, 256, -1, 0, native.MOE_ERR_INVALID_ARG, "M ="),
    (16, 256, 17, 1, native.MOE_ERR_UNSUPPORTED, "exceeds"),
    (16, 256, 2, 1, native.MOE_ERR_INVALID_ARG, "aligned"),  # null pointers
])
def test_gemv_rejects_bad_arguments_before_the_gpu(L, rows, k, M, engine, status, frag):
    assert L.moe_gemv(None, None, None, rows, k, M, engine, None) == status
    assert frag in native.last_error()


def test_gemv_zero_tokens_and_pack_checks(L):
    assert L.moe_gemv(None, None, None, 16, 256, 0, 0, None) == native.MOE_OK
    assert L.moe_gemv_pack(None, None, 16, 64, None) == native.MOE_ERR_INVALID_ARG
    assert L.moe_gemv_pack(ctypes.c_void_p(24), ctypes.c_void_p(32), 16, 64, None) == native.MOE_ERR_INVALID_ARG
    assert "aligned" in native.last_error()
    assert L.moe_gemv_pack(ctypes.c_void_p(16), ctypes.c_void_p(32), 15, 64, None) == native.MOE_ERR_INVALID_ARG


def test_new_entry_points_reject_bad_arguments_before_the_gpu(L):
    p = ctypes.c_void_p
    assert L.moe_set_grid(None, 0) == native.MOE_ERR_INVALID_ARG
    assert L.moe_set_wait_limit(None, 0) == native.MOE_ERR_INVALID_ARG
    assert L.moe_combine_partials(None, 2, 16, None, None) == native.MOE_ERR_INVALID_ARG
    assert L.moe_combine_partials(p(16), 2, 18, p(4096), None) == native.MOE_ERR_INVALID_ARG   # n % 4
    assert L.moe_combine_partials(p(16), 0, 16, p(4096), None) == native.MOE_ERR_INVALID_ARG   # no parts
    assert L.moe_combine_partials(p(20), 2, 16, p(4096), None) == native.MOE_ERR_INVALID_ARG   # misaligned
    assert "aligned" in native.last_error()
    assert L.moe_combine_partials(p(16), 2, 16, p(32), None) == native.MOE_ERR_INVALID_ARG     # overlap
    assert "overlaps" in native.last_error()
    assert L.moe_combine_partials(p(16), 2, 0, p(4096), None) == native.MOE_OK                 # nothing to do
    assert L.moe_route_static_read_status(None, None) == native.MOE_ERR_INVALID_ARG
    assert L.moe_route_static_read_status(p(2), None) == native.MOE_ERR_INVALID_ARG            # misaligned


def test_info_struct_matches_the_header():
    """moe_info_t's fields, in order, as the header declares them."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    end = src.index("} moe_info_t;")
    body = src[src.rindex("typedef struct {", 0, end) + len("typedef struct {"):end]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if decl:
            names += [n.strip() for n in decl.split(None, 1)[1].split(",")] if not decl.startswith("unsigned long long") \
                else [n.strip() for n in decl[len("unsigned long long"):].split(",")]
    assert names == [f for f, _ in native.moe_info_t._fields_]
