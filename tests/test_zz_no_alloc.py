"""GPU test of moe_route_static, the routing entry point that allocates nothing.

Callers that cannot call cudaMalloc (code running while someone else captures
a CUDA graph, allocators that forbid outside allocations, paths that must not
risk an allocation failure) route tokens through moe_route_static, whose
scratch is a fixed array inside the library.  Its routing must equal what the
layer's own forward computes, call after call, although every call reuses
the same scratch.  This file sorts last so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

from weight_streaming_expert_gb300 import native
from weight_streaming_expert_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _route_static():
    f = native.lib().moe_route_static
    vp, ci = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [ci, ci, ci, vp, vp, vp, ci, vp, vp, vp]
    f.restype = ci
    return f


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_static_routing_equals_layer_routing_on_consecutive_calls():
    from weight_streaming_expert_gb300 import MoELayer
    shape = wl.LayerShape(hidden=2560, n_experts=512, topk=8, inter=128)
    w_r, w_gu, w_d = wl.layer_weights(shape, seed=77, device=DEV)
    layer = MoELayer(w_r, w_gu, w_d, topk=shape.topk)
    route = _route_static()
    stream = torch.cuda.current_stream()
    zipf = wl.zipf_router_bias(shape.n_experts).to(DEV)
    # two calls in a row through the same scratch: uniform M=6, then a
    # biased (skewed) M=16 block
    for call, (M, bias) in enumerate(((6, None), (16, zipf))):
        layer.set_router_bias(bias)
        x = wl.tokens(M, shape.hidden, seed=900 + call, device=DEV)
        tw_ref = torch.empty((M, shape.topk), dtype=torch.float32, device=DEV)
        _, idx_ref = layer(x, topk_w=tw_ref)
        idx = torch.full((M, shape.topk), -1, dtype=torch.int32, device=DEV)
        tw = torch.full((M, shape.topk), -1.0, dtype=torch.float32, device=DEV)
        rc = route(shape.hidden, shape.n_experts, shape.topk, _p(x), _p(w_r), _p(bias), M,
                   _p(idx), _p(tw), ctypes.c_void_p(stream.cuda_stream))
        assert rc == native.MOE_OK, native.last_error()
        torch.cuda.synchronize()
        # same matvec split, summation order and top-k code as the layer kernel
        assert torch.equal(idx, idx_ref), f"call {call}: expert ids differ"
        assert torch.equal(tw, tw_ref), f"call {call}: weights differ"
    layer.close()


def test_static_routing_rejects_sizes_beyond_its_scratch():
    route = _route_static()
    x = torch.zeros((17, 256), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((16, 256), dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros((17, 2), dtype=torch.int32, device=DEV)
    rc = route(256, 16, 2, _p(x), _p(w), None, 17, _p(idx), None, None)
    assert rc == native.MOE_ERR_UNSUPPORTED
    assert "16 tokens" in native.last_error()
    rc = route(256, 2048, 2, _p(x), _p(w), None, 1, _p(idx), None, None)
    assert rc == native.MOE_ERR_UNSUPPORTED
