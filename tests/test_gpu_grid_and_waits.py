"""GPU tests of the layer kernel's grid and of its bounded waits.

* Grid: the layer kernel's CTAs wait on one another, so all must be
  resident; a caller that leaves SMs to other work (a collective on another
  stream) launches the layer on fewer CTAs (moe_set_grid).  The work is split
  over gridDim, so every grid gives the same bits, and the oracle's answer.
* Bounded waits: a test-only flag makes one CTA leave out one grid-wide
  arrival; with a short wait limit the dependent waits run out, the call
  returns, moe_get_status reports MOE_ERR_DEVICE_TIMEOUT with the phase that
  gave up, and the next call is exact again.  Nothing faults, traps or hangs:
  every wait ends at its limit.
"""
import time

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
def MoELayer():
    from weight_streaming_expert_gb300 import MoELayer as L
    return L


@pytest.fixture(scope="module")
def ling(MoELayer):
    w_r, w_gu, w_d = wl.layer_weights(wl.LING, seed=1000, device=DEV)
    layer = MoELayer(w_r, w_gu, w_d, topk=wl.LING.topk)
    host = dict(wr=bits(w_r), wgu=bits(w_gu), wd=bits(w_d))
    del w_r, w_gu, w_d
    torch.cuda.empty_cache()
    yield layer, host
    layer.set_grid(0)
    layer.close()


CASES = [(6, 1, False), (1, 2, False), (16, 3, True), (64, 4, False)]


def test_full_grid_is_one_cta_per_sm(ling):
    layer, _ = ling
    info = layer.info()
    assert info.grid_ctas == info.n_sms == torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("ctas", [148, 120, 64])
def test_smaller_grids_match_the_oracle_and_the_full_grid(oracle, ling, ctas):
    layer, host = ling
    ref = []
    layer.set_grid(0)
    for M, seed, zipf in CASES:
        layer.set_router_bias(wl.zipf_router_bias(wl.LING.n_experts) if zipf else None)
        x = wl.tokens(M, wl.LING.hidden, seed=9_000_000 + seed, device=DEV)
        out, idx = layer(x)
        ref.append((x, out.clone(), idx.clone()))
    torch.cuda.synchronize()
    layer.set_grid(ctas)
    assert layer.info().grid_ctas == ctas
    # PDL-chained calls on one stream, no host synchronisation between them
    got = []
    for (M, seed, zipf), (x, _, _) in zip(CASES, ref):
        layer.set_router_bias(wl.zipf_router_bias(wl.LING.n_experts) if zipf else None)
        got.append(layer(x))
    torch.cuda.synchronize()
    assert layer.status() == 0
    for (M, seed, zipf), (x, ro, ri), (o, i) in zip(CASES, ref, got):
        assert torch.equal(i, ri), f"M={M}: expert ids differ from the full grid's"
        assert torch.equal(o.view(torch.int16), ro.view(torch.int16)), f"M={M}: outputs differ"
    # and the oracle on two of them (the rest are bit-equal to full-grid calls
    # that the other parity tests hold to the oracle)
    for (M, seed, zipf), (x, _, _), (o, i) in list(zip(CASES, ref, got))[:2]:
        parity.check_layer(oracle, bits(x), host["wr"], host["wgu"], host["wd"], wl.LING.topk,
                           o.float().cpu().numpy(), i.cpu().numpy())
    layer.set_router_bias(None)
    layer.set_grid(0)


def test_topk_exchange_both_parities_and_a_tiny_grid(ling):
    """Calls of more tokens than a CTA has warps find each token's top-k once
    in the grid and exchange the slots through a buffer of the call's parity,
    which the call clears after use.  Chained calls that take the exchange on
    both parities, with M changing, equal the same calls made alone; on a
    4-CTA grid every warp takes several tokens and the results stay the
    same bits."""
    layer, _ = ling
    layer.set_router_bias(None)
    Ms = [11, 40, 2, 64, 33, 16, 64, 12]
    xs = [wl.tokens(M, wl.LING.hidden, seed=7_700_000 + i, device=DEV) for i, M in enumerate(Ms)]
    alone = []
    for x in xs:
        out, idx = layer(x)
        torch.cuda.synchronize()
        alone.append((out.clone(), idx.clone()))
    chained = [layer(x) for x in xs]
    torch.cuda.synchronize()
    assert layer.status() == 0
    for n, ((o, i), (ro, ri)) in enumerate(zip(chained, alone)):
        assert torch.equal(i, ri), f"call {n} (M = {Ms[n]}): expert ids differ"
        assert torch.equal(o.view(torch.int16), ro.view(torch.int16)), f"call {n} (M = {Ms[n]}): outputs differ"
    layer.set_grid(4)
    try:
        small = [layer(xs[n]) for n in (3, 4)]
        torch.cuda.synchronize()
        assert layer.status() == 0
        for (o, i), n in zip(small, (3, 4)):
            assert torch.equal(i, alone[n][1]), f"4 CTAs, M = {Ms[n]}: expert ids differ"
            assert torch.equal(o.view(torch.int16), alone[n][0].view(torch.int16)), f"4 CTAs, M = {Ms[n]}"
    finally:
        layer.set_grid(0)


def test_grid_bounds_are_checked(ling):
    from weight_streaming_expert_gb300 import native as N
    layer, _ = ling
    n = layer.info().n_sms
    with pytest.raises(N.MoEError):
        layer.set_grid(n + 1)
    with pytest.raises(N.MoEError):
        layer.set_grid(-1)
    assert layer.info().grid_ctas == n


@pytest.mark.parametrize("M", [1, 6])
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_exact(MoELayer, M):
    from weight_streaming_expert_gb300 import native as N
    shape = wl.LayerShape(hidden=1024, n_experts=64, topk=4, inter=256)
    w_r, w_gu, w_d = (t.to(DEV) for t in wl.layer_weights(shape, seed=21))
    clean = MoELayer(w_r, w_gu, w_d, topk=4)
    layer = MoELayer(w_r, w_gu, w_d, topk=4)
    limit_ns = 2_000_000                       # 2 ms instead of 2 s
    layer.set_wait_limit(limit_ns)
    assert layer.info().wait_limit_ns == limit_ns
    xs = [wl.tokens(M, shape.hidden, seed=60 + i, device=DEV) for i in range(3)]
    want = [clean(x) for x in xs]
    torch.cuda.synchronize()
    assert clean.status() == 0
    # a normal call, then one whose static-tile count is one arrival short
    layer(xs[0])
    torch.cuda.synchronize()
    assert layer.status() == N.MOE_OK
    t0 = time.perf_counter()
    layer(xs[1], test_skip_arrival=True)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert dt < 1.0, f"the injected call took {dt:.3f} s: the wait limit was not applied"
    st = layer.status()
    msg = N.last_error()
    assert st == N.MOE_ERR_DEVICE_TIMEOUT, (st, msg)
    # every publisher's grid-wide wait on the short count gave up (bit 16);
    # the first wait recorded is that one (phase 2) or a producer's wait for
    # the readiness it would have signalled (phase 3)
    import re
    bits_set = int(re.search(r"device status bits 0x([0-9a-f]+)", msg).group(1), 16)
    assert bits_set & 16, msg
    assert re.search(r"first timeout: phase [23] ", msg), msg
    # the status read restarted the counts: the next calls are exact again
    for x, (wo, wi) in zip(xs, want):
        o, i = layer(x)
        torch.cuda.synchronize()
        assert torch.equal(i, wi) and torch.equal(o.view(torch.int16), wo.view(torch.int16))
    assert layer.status() == N.MOE_OK
    layer.set_wait_limit(0)
    assert layer.info().wait_limit_ns == 2_000_000_000
    layer.close()
    clean.close()
