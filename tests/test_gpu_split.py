"""GPU tests of the tensor-parallel split of the layer (the post's TP4: each
GPU holds a quarter of every expert's intermediate rows, routes every token,
and the MoE chain ends in an all-reduce of the partial outputs).

On one GPU the G slices run one after another as layers of their own; each
writes its combine unrounded (MOE_FWD_OUT_F32), moe_combine_partials sums the
G parts in order and rounds once, and the result must match the oracle's
UNSPLIT layer under the same rule as every other output (routing bit-exact up
to near-ties, max-abs <= 2e-2, rel-L2 <= 1e-2).
"""
import numpy as np
import pytest
import torch

from tests import parity
from weight_streaming_expert_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def bits(t):
    return wl.bf16_bits(t)


@pytest.fixture(scope="module")
def lib():
    from weight_streaming_expert_gb300 import layer
    return layer


def split_layers(lib, w_r, w_gu, w_d, k, G):
    layers = []
    for r in range(G):
        gu, d = lib.tp_slice(w_gu, w_d, r, G)
        layers.append(lib.MoELayer(w_r, gu, d, topk=k))
        del gu, d
    return layers


def run_split(lib, layers, x, bias=None):
    """Every slice on the same tokens, fp32 parts gathered side by side,
    then the ordered sum with one rounding."""
    M, H = x.shape
    parts = torch.empty((len(layers), M, H), dtype=torch.float32, device=DEV)
    idxs = []
    for g, layer in enumerate(layers):
        layer.set_router_bias(bias)
        _, idx = layer(x, out=parts[g], out_f32=True)
        idxs.append(idx)
    out = lib.combine_partials(parts)
    torch.cuda.synchronize()
    for layer in layers:
        assert layer.status() == 0
    return out, idxs, parts


def test_fp32_output_is_the_combine_before_its_rounding(lib, oracle):
    """The fp32 mode writes exactly what the bf16 mode rounds."""
    shape = wl.LayerShape(hidden=1280, n_experts=40, topk=3, inter=256)
    w_r, w_gu, w_d = wl.layer_weights(shape, seed=31)
    layer = lib.MoELayer(w_r.to(DEV), w_gu.to(DEV), w_d.to(DEV), topk=3)
    for M in (1, 6, 13, 64):
        x = wl.tokens(M, shape.hidden, seed=40 + M).to(DEV)
        o16, i16 = layer(x)
        o32, i32 = layer(x, out_f32=True)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(i16, i32)
        assert torch.equal(o32.to(torch.bfloat16).view(torch.int16), o16.view(torch.int16))
        # against the oracle's fp32 combine (before its own rounding)
        ref = oracle.moe_forward(bits(x.cpu()), bits(w_r), bits(w_gu), bits(w_d), 3)
        if np.array_equal(i16.cpu().numpy(), ref["idx"]):
            got, want = o32.cpu().numpy().astype(np.float64), ref["acc"].astype(np.float64)
            assert np.abs(got - want).max() <= parity.MAX_ABS
            assert np.linalg.norm(got - want) / np.linalg.norm(want) <= parity.MAX_REL_L2
    layer.close()


def test_combine_partials_order_and_rounding(lib):
    """Ordered fp32 sum, one round-to-nearest-even to bf16, for 1..8 parts."""
    g = torch.Generator().manual_seed(5)
    for G in (1, 2, 3, 4, 8):
        parts = torch.randn((G, 7, 256), generator=g) * 3
        parts[:, 0, :8] = torch.tensor([1.0, 2 ** -9, -2 ** -9, 3e-39, -0.0, 1e30, -1e30, 2 ** -8])[None, :]
        want = parts[0].clone()
        for p in range(1, G):
            want = want + parts[p]            # fp32, in part order
        got = lib.combine_partials(parts.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(got.cpu().view(torch.int16), want.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("H,E,k,I,G,M", [(1280, 40, 3, 512, 4, 13), (512, 64, 6, 256, 2, 5),
                                         (2560, 24, 2, 512, 4, 64), (256, 16, 2, 256, 2, 1)])
def test_split_small_layers_match_the_unsplit_oracle(lib, oracle, H, E, k, I, G, M):
    shape = wl.LayerShape(hidden=H, n_experts=E, topk=k, inter=I)
    w_r, w_gu, w_d = wl.layer_weights(shape, seed=H + E + G)
    layers = split_layers(lib, w_r.to(DEV), w_gu.to(DEV), w_d.to(DEV), k, G)
    x = wl.tokens(M, H, seed=M + G).to(DEV)
    out, idxs, _ = run_split(lib, layers, x)
    for i in idxs[1:]:
        assert torch.equal(i, idxs[0])        # every slice routes alike
    parity.check_layer(oracle, bits(x.cpu()), bits(w_r), bits(w_gu), bits(w_d), k,
                       out.float().cpu().numpy(), idxs[0].cpu().numpy())
    for layer in layers:
        layer.close()


@pytest.fixture(scope="module")
def ling_split(lib):
    """The Ling-shaped layer of seed 1000 split four ways (inter 512 -> 4 x 128)."""
    w_r, w_gu, w_d = wl.layer_weights(wl.LING, seed=1000, device=DEV)
    layers = split_layers(lib, w_r, w_gu, w_d, wl.LING.topk, 4)
    host = dict(wr=bits(w_r), wgu=bits(w_gu), wd=bits(w_d))
    del w_r, w_gu, w_d
    torch.cuda.empty_cache()
    yield layers, host
    for layer in layers:
        layer.close()


@pytest.mark.parametrize("M,zipf", [(1, False), (6, False), (16, True)])
def test_ling_split_four_ways_matches_the_unsplit_oracle(lib, oracle, ling_split, M, zipf):
    layers, host = ling_split
    bias = wl.zipf_router_bias(wl.LING.n_experts) if zipf else None
    x = wl.tokens(M, wl.LING.hidden, seed=8_000_000 + M, device=DEV)
    out, idxs, parts = run_split(lib, layers, x, bias=bias)
    for i in idxs[1:]:
        assert torch.equal(i, idxs[0])
    st = parity.check_layer(oracle, bits(x), host["wr"], host["wgu"], host["wd"], wl.LING.topk,
                            out.float().cpu().numpy(), idxs[0].cpu().numpy(),
                            bias=None if bias is None else bias.numpy())
    # the parts sum to the oracle's unrounded combine of the unsplit layer
    if st["near_tie_tokens"] == 0:
        got = parts.sum(dim=0).cpu().numpy().astype(np.float64)
        want = st["ref"]["acc"].astype(np.float64)
        assert np.abs(got - want).max() <= parity.MAX_ABS
        assert np.linalg.norm(got - want) / np.linalg.norm(want) <= parity.MAX_REL_L2
    for layer in layers:
        layer.set_router_bias(None)


def test_combine_partials_rejects_bad_arguments(lib):
    from weight_streaming_expert_gb300 import native as N
    L = N.lib()
    parts = torch.zeros((2, 4, 8), dtype=torch.float32, device=DEV)
    out = torch.zeros((4, 8), dtype=torch.bfloat16, device=DEV)
    import ctypes
    p = ctypes.c_void_p
    assert L.moe_combine_partials(p(parts.data_ptr()), 2, 30, p(out.data_ptr()), None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_combine_partials(p(parts.data_ptr() + 4), 2, 32, p(out.data_ptr()), None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_combine_partials(p(parts.data_ptr()), 0, 32, p(out.data_ptr()), None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_combine_partials(p(parts.data_ptr()), 2, 32, p(parts.data_ptr()), None) == N.MOE_ERR_INVALID_ARG
    assert "overlaps" in N.last_error()
