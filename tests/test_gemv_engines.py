"""The expert contraction on both engines (include/gemv.h) against its plain
definition, y[m][r] = sum_k W[r][k] x[m][k], evaluated in float64 on the
CPU over the same bf16 values.  Sizes span several tiles, ragged token
counts and every token count the engines are compiled for."""
import numpy as np
import pytest
import torch

from weight_streaming_expert_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def reference(w, x):
    return x.double().numpy() @ w.double().numpy().T


@pytest.mark.parametrize("rows,k", [(8, 256), (264, 768), (1024, 2560), (2560, 512), (40, 3072)])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 7, 8, 9, 13, 16])
@pytest.mark.parametrize("engine", ["cuda_cores", "tensor_cores"])
def test_gemv_matches_definition(rows, k, M, engine):
    from weight_streaming_expert_gb300 import gemv as G
    g = torch.Generator().manual_seed(rows * 131 + k * 7 + M)
    w = (torch.randn(rows, k, generator=g) * wl.WEIGHT_STD).to(torch.bfloat16)
    x = torch.randn(M, k, generator=g).to(torch.bfloat16)
    packed = G.pack(w.to(DEV))
    y = G.gemv(packed, x.to(DEV), G.CUDA_CORES if engine == "cuda_cores" else G.TENSOR_CORES)
    torch.cuda.synchronize()
    ref = reference(w, x)
    got = y.cpu().double().numpy()
    # fp32 sums of k products: |error| <= k * 2^-23 * sum |w x| (loose), far
    # below any mistake in an index or an operand
    bound = k * 2.0 ** -23 * (np.abs(w.double().numpy()) @ np.abs(x.double().numpy()).T).T + 1e-30
    assert got.shape == ref.shape
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


def test_engines_agree_on_the_expert_shape():
    """Gate/up shape of one Ling-shaped expert (1024 x 2560) at M = 6."""
    from weight_streaming_expert_gb300 import gemv as G
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(1024, 2560, generator=g) * wl.WEIGHT_STD).to(torch.bfloat16).to(DEV)
    x = torch.randn(6, 2560, generator=g).to(torch.bfloat16).to(DEV)
    packed = G.pack(w)
    a = G.gemv(packed, x, G.CUDA_CORES)
    b = G.gemv(packed, x, G.TENSOR_CORES)
    torch.cuda.synchronize()
    assert torch.allclose(a, b, rtol=1e-4, atol=1e-4)


def test_gemv_rejects_bad_arguments():
    from weight_streaming_expert_gb300 import gemv as G
    from weight_streaming_expert_gb300 import native
    w = torch.zeros(16, 256, dtype=torch.bfloat16, device=DEV)
    packed = G.pack(w)
    x = torch.zeros(17, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(native.MoEError) as e:
        G.gemv(packed, x, G.TENSOR_CORES)
    assert e.value.status == native.MOE_ERR_UNSUPPORTED
    with pytest.raises(native.MoEError) as e:
        G.gemv(packed, x[:4], 7)
    assert e.value.status == native.MOE_ERR_INVALID_ARG
    assert G.gemv(packed, x[:0], G.CUDA_CORES).shape == (0, 16)
    assert G.status() == native.MOE_OK
