"""GPU tests of the vocabulary projection (include/lm_head.h) against the CPU
oracle: logits[m][v] = x[m] . W[v], fp32 over bf16.  The GPU sums in another
order than the oracle's ascending one, so each logit may differ by the fp32
summation bound 1e-5 * sum_k |x_k w_k| (+ 1e-6), the bound the oracle itself
is pinned to against a float64 matmul."""
import numpy as np
import pytest
import torch

from weight_streaming_expert_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def bits(t):
    return wl.bf16_bits(t.cpu())


def f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.fixture(scope="module")
def LmHead():
    from weight_streaming_expert_gb300 import LmHead as L
    return L


def check(oracle, x, w, got):
    xb, wb = bits(x), bits(w)
    want = oracle.lm_head(xb, wb)
    bound = 1e-5 * (np.abs(f32(xb)) @ np.abs(f32(wb)).T) + 1e-6
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(err <= bound), f"max err {err.max():.3g} (bound there {bound.flat[err.argmax()]:.3g})"


@pytest.mark.parametrize("H,V,M", [(256, 333, 1), (256, 333, 5), (256, 333, 16), (512, 1000, 3),
                                   (1280, 77, 16), (4096, 1025, 2), (2560, 8, 1), (1024, 9, 7)])
def test_small_shapes_match_oracle(oracle, LmHead, H, V, M):
    w = wl.lm_head_weight(V, H, seed=H + V).to(DEV)
    x = wl.tokens(M, H, seed=M + 40).to(DEV)
    head = LmHead(w)
    got = head(x)
    torch.cuda.synchronize()
    assert head.status() == 0
    check(oracle, x, w, got.cpu().numpy())
    head.close()


def test_full_vocabulary(oracle, LmHead):
    """The model's projection: hidden 2560 x 157,184 rows, M = 6."""
    H, V = 2560, wl.LM_HEAD_VOCAB
    w = wl.lm_head_weight(V, H, seed=4000, device=DEV)
    x = wl.tokens(6, H, seed=4001, device=DEV)
    head = LmHead(w)
    got = head(x)
    torch.cuda.synchronize()
    assert head.status() == 0
    check(oracle, x, w, got.cpu().numpy())
    head.close()


def test_graph_replay_equals_eager(LmHead):
    H, V = 2560, 40000
    w = wl.lm_head_weight(V, H, seed=4100, device=DEV)
    x = wl.tokens(4, H, seed=4101, device=DEV)
    head = LmHead(w)
    eager = head(x).clone()
    s = torch.cuda.Stream()
    out = torch.empty_like(eager)
    with torch.cuda.stream(s):
        head(x, out, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                head(x, out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    head.close()


def test_zero_token_and_arguments(LmHead):
    from weight_streaming_expert_gb300 import native as N
    H, V = 512, 100
    w = wl.lm_head_weight(V, H, seed=7, device=DEV)
    head = LmHead(w)
    out = head(torch.zeros((2, H), dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert not torch.any(out)
    L = N.lib()
    x = torch.zeros((17, H), dtype=torch.bfloat16, device=DEV)
    lg = torch.empty((17, V), dtype=torch.float32, device=DEV)
    import ctypes
    p = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    assert L.moe_lm_head_forward(head._h, p(x), p(lg), 17, None) == N.MOE_ERR_UNSUPPORTED
    assert L.moe_lm_head_forward(head._h, p(x, 2), p(lg), 1, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_lm_head_forward(head._h, None, p(lg), 1, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_lm_head_forward(head._h, p(x), p(lg), 0, None) == N.MOE_OK
    assert L.moe_lm_head_forward(None, p(x), p(lg), 1, None) == N.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert head.status() == 0
    head.close()
