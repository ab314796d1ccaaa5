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

import numpy as np
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


_W = {}


def _router(E, H=2560):
    """One router weight per expert count, kept for the module."""
    if E not in _W:
        g = torch.Generator().manual_seed(1234 + E)
        _W[E] = (torch.randn((E, H), generator=g) * wl.WEIGHT_STD).to(torch.bfloat16)
    return _W[E]


@pytest.mark.parametrize("E", [17, 512, 1000])
@pytest.mark.parametrize("k", [1, 8, 32])
@pytest.mark.parametrize("M", [1, 6, 16])
@pytest.mark.parametrize("with_bias", [False, True])
def test_static_routing_matches_the_oracle(oracle, E, k, M, with_bias):
    """Expert ids bit-exact against the oracle's router and top-k (up to the
    documented near-ties), weights within a few fp32 ulps, and a clean status
    word read back through moe_route_static_read_status."""
    if k > E:
        pytest.skip("k > E is refused")
    from tests import parity
    H = 2560
    w = _router(E, H)
    x = wl.tokens(M, H, seed=70 + M + E)
    bias = None
    if with_bias:
        bias = torch.from_numpy((np.random.default_rng(E + k).standard_normal(E) * 0.5).astype(np.float32))
    route = _route_static()
    wd, xd = w.to(DEV), x.to(DEV)
    bd = None if bias is None else bias.to(DEV)
    idx = torch.full((M, k), -1, dtype=torch.int32, device=DEV)
    tw = torch.full((M, k), -1.0, dtype=torch.float32, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    rc = route(H, E, k, _p(xd), _p(wd), _p(bd), M, _p(idx), _p(tw), sp)
    assert rc == native.MOE_OK, native.last_error()
    assert native.lib().moe_route_static_read_status(_p(status), sp) == native.MOE_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    logits = oracle.router_logits(wl.bf16_bits(x), wl.bf16_bits(w), None if bias is None else bias.numpy())
    ref_idx, ref_w = oracle.topk_softmax(logits, k)
    gi, gw = idx.cpu().numpy(), tw.cpu().numpy()
    for m in range(M):
        assert parity.routing_ok(gi[m], ref_idx[m], logits[m]), f"token {m}: {gi[m]} vs {ref_idx[m]}"
        want = ref_w[m] if np.array_equal(gi[m], ref_idx[m]) else oracle.weights_for_set(logits[m], gi[m])
        # the GPU's logits differ from the oracle's by fp32 summation order
        # (~3e-6 for a 2560-term dot of this scale); a weight exp(l_j - l_0) / S
        # moves by a few times that, relatively
        np.testing.assert_allclose(gw[m], want, rtol=1e-4, atol=1e-6)
        assert abs(float(gw[m].sum()) - 1.0) <= 1e-5


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
    assert native.lib().moe_route_static_read_status(None, None) == native.MOE_ERR_INVALID_ARG
