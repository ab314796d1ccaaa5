"""GPU parity tests: the CUDA path (through the C ABI) against the CPU oracle.

Every case compares routing indices (bit-exact up to documented near-ties)
and outputs (max-abs <= 2e-2 and rel-L2 <= 1e-2) element by element on the
same seeded inputs.  Sizes span several tiles and ragged tails; the full
hidden-2560 / 512-expert / top-8 / inter-512 layer is run at M = 1, 6, 16
and across the sweep M in {2,4,8,32,64} x {uniform, Zipf}.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests import parity
from tests.test_golden import load_tiny_golden
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
    """One full-size layer (seed 1000) shared by the full-size cases."""
    w_r, w_gu, w_d = wl.layer_weights(wl.LING, seed=1000, device=DEV)
    layer = MoELayer(w_r, w_gu, w_d, topk=wl.LING.topk)
    host = dict(wr=bits(w_r), wgu=bits(w_gu), wd=bits(w_d))
    del w_r, w_gu, w_d
    torch.cuda.empty_cache()
    yield layer, host
    layer.close()


def run_and_check(orc, layer, host, x, k, bias=None, **kw):
    layer.set_router_bias(bias)
    out, idx = layer(x)
    torch.cuda.synchronize()
    st = layer.status()
    if st != 0:
        from weight_streaming_expert_gb300 import native
        raise AssertionError(f"device status {st}: {native.last_error()}")
    st = parity.check_layer(orc, bits(x), host["wr"], host["wgu"], host["wd"], k,
                            out.float().cpu().numpy(), idx.cpu().numpy(),
                            bias=None if bias is None else bias.cpu().numpy(), **kw)
    return out, idx, st


def small_layer(MoELayer, shape, seed):
    w_r, w_gu, w_d = wl.layer_weights(shape, seed=seed, device="cpu")
    layer = MoELayer(w_r.to(DEV), w_gu.to(DEV), w_d.to(DEV), topk=shape.topk)
    return layer, dict(wr=bits(w_r), wgu=bits(w_gu), wd=bits(w_d))


# ------------------------------------------------------------ small layer --

def test_tiny_layer_matches_oracle_and_golden(oracle, MoELayer):
    """The small oracle-check layer, seed 0, M = 1 and M = 4."""
    recs = load_tiny_golden()
    for M in (1, 4):
        w_r, w_gu, w_d, x = wl.tiny_case(M=M, seed=0)
        layer = MoELayer(w_r.to(DEV), w_gu.to(DEV), w_d.to(DEV), topk=wl.TINY.topk)
        host = dict(wr=bits(w_r), wgu=bits(w_gu), wd=bits(w_d))
        out, idx, st = run_and_check(oracle, layer, host, x.to(DEV), wl.TINY.topk)
        assert st["near_tie_tokens"] == 0
        assert np.array_equal(idx.cpu().numpy().ravel(), recs[M]["idx"])
        got = out.float().cpu().numpy().ravel()
        want = parity.bf16_bits_to_f32(recs[M]["out"])
        assert np.abs(got - want).max() <= parity.MAX_ABS
        layer.close()


@pytest.mark.parametrize("M", [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 48, 63, 64])
def test_tiny_layer_all_M(oracle, MoELayer, M):
    layer, host = small_layer(MoELayer, wl.TINY, seed=11)
    x = wl.tokens(M, wl.TINY.hidden, seed=100 + M).to(DEV)
    run_and_check(oracle, layer, host, x, wl.TINY.topk)
    layer.close()


RAGGED = [
    # (hidden, n_experts, topk, inter, M): every hidden/256 and inter the kernels
    # are built for, expert counts off the warp width, k = 1 and k = 32
    (1280, 40, 3, 256, 13),
    (512, 1000, 1, 128, 7),
    (256, 64, 32, 128, 5),
    (1024, 96, 6, 512, 64),
    (4096, 128, 4, 256, 3),
    (3072, 33, 5, 128, 11),
    (2048, 17, 17, 512, 2),
    (2560, 24, 2, 512, 23),
    (1024, 700, 3, 256, 19),  # more tokens than warps with E > 512: one token per warp at a time
]


@pytest.mark.parametrize("H,E,k,I,M", RAGGED)
def test_ragged_shapes(oracle, MoELayer, H, E, k, I, M):
    shape = wl.LayerShape(hidden=H, n_experts=E, topk=k, inter=I)
    layer, host = small_layer(MoELayer, shape, seed=H + E + k)
    x = wl.tokens(M, H, seed=7 * M + 1).to(DEV)
    run_and_check(oracle, layer, host, x, k)
    layer.close()


def test_a_later_smaller_handle_keeps_the_earlier_one_launchable(oracle, MoELayer):
    """Two handles that run the same kernel instance (same hidden size) with
    different shared-memory needs (1000 experts need a larger routing area
    than 16): the instance's dynamic shared-memory limit is a property of the
    kernel function, so creating the smaller handle second must not make the
    larger one's launches fail."""
    big_shape = wl.LayerShape(hidden=256, n_experts=1000, topk=2, inter=128)
    big, host = small_layer(MoELayer, big_shape, seed=41)
    small, small_host = small_layer(MoELayer, wl.LayerShape(hidden=256, n_experts=16, topk=2, inter=128), seed=42)
    assert big.info().smem_bytes > small.info().smem_bytes
    for M in (3, 12):
        run_and_check(oracle, big, host, wl.tokens(M, 256, seed=4100 + M).to(DEV), 2)
        run_and_check(oracle, small, small_host, wl.tokens(M, 256, seed=4200 + M).to(DEV), 2)
    small.close()
    big.close()


def test_uniform_logits_tie_rule(oracle, MoELayer):
    """W_r = 0: every logit ties, so experts 0..k-1 in order with w = 1/k."""
    shape = wl.LayerShape(hidden=512, n_experts=64, topk=4, inter=128)
    w_r, w_gu, w_d = wl.layer_weights(shape, seed=5)
    w_r = torch.zeros_like(w_r)
    layer = MoELayer(w_r.to(DEV), w_gu.to(DEV), w_d.to(DEV), topk=4)
    x = wl.tokens(9, 512, seed=9).to(DEV)
    tw = torch.empty((9, 4), dtype=torch.float32, device=DEV)
    out, idx = layer(x, topk_w=tw)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(4, dtype=np.int32), (9, 1)))
    assert np.all(tw.cpu().numpy() == np.float32(0.25))
    ref = oracle.moe_forward(bits(x.cpu()), bits(w_r), bits(w_gu), bits(w_d), 4)
    mx, rel = parity.compare_outputs(out.float().cpu().numpy(), ref["out"])
    assert mx <= parity.MAX_ABS and rel <= parity.MAX_REL_L2
    layer.close()


def test_zero_input_gives_zero_output(MoELayer):
    layer, _ = small_layer(MoELayer, wl.TINY, seed=3)
    x = torch.zeros((5, wl.TINY.hidden), dtype=torch.bfloat16, device=DEV)
    out, idx = layer(x)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out.float()).item() == 0
    assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(wl.TINY.topk, dtype=np.int32), (5, 1)))
    layer.close()


def test_identical_tokens_identical_rows(MoELayer):
    layer, _ = small_layer(MoELayer, wl.TINY, seed=4)
    x = wl.tokens(1, wl.TINY.hidden, seed=4).repeat(20, 1).contiguous().to(DEV)
    out, idx = layer(x)
    torch.cuda.synchronize()
    o = out.cpu()
    assert all(torch.equal(o[0], o[i]) for i in range(1, 20))
    assert all(torch.equal(idx[0], idx[i]) for i in range(1, 20))
    layer.close()


# ------------------------------------------------------------- full size --

@pytest.mark.parametrize("M,seed,zipf", [(6, 1, False), (6, 2, False), (1, 3, False), (16, 4, True),
                                         (16, 5, False), (1, 6, True)])
def test_ling_layer(oracle, ling, M, seed, zipf):
    layer, host = ling
    bias = wl.zipf_router_bias(wl.LING.n_experts) if zipf else None
    x = wl.tokens(M, wl.LING.hidden, seed=1_000_000 + seed, device=DEV)
    run_and_check(oracle, layer, host, x, wl.LING.topk, bias=bias)


@pytest.mark.parametrize("M", [2, 4, 8, 32, 64])
@pytest.mark.parametrize("zipf", [False, True])
def test_ling_sweep(oracle, ling, M, zipf):
    layer, host = ling
    bias = wl.zipf_router_bias(wl.LING.n_experts) if zipf else None
    x = wl.tokens(M, wl.LING.hidden, seed=2_000_000 + M + (7 if zipf else 0), device=DEV)
    run_and_check(oracle, layer, host, x, wl.LING.topk, bias=bias)


@pytest.fixture(scope="module")
def ling_tp4(MoELayer):
    """The per-GPU slice of a 4-way TP split of the Ling-shaped layer (inter
    512 / 4 = 128 rows of every expert), full size, seed 1100."""
    w_r, w_gu, w_d = wl.layer_weights(wl.LING_TP4, seed=1100, device=DEV)
    layer = MoELayer(w_r, w_gu, w_d, topk=wl.LING_TP4.topk)
    host = dict(wr=bits(w_r), wgu=bits(w_gu), wd=bits(w_d))
    del w_r, w_gu, w_d
    torch.cuda.empty_cache()
    yield layer, host
    layer.close()


@pytest.mark.parametrize("M,seed,zipf", [(6, 11, False), (1, 12, False), (16, 13, True), (64, 14, False)])
def test_ling_tp4_slice(oracle, ling_tp4, M, seed, zipf):
    layer, host = ling_tp4
    bias = wl.zipf_router_bias(wl.LING_TP4.n_experts) if zipf else None
    x = wl.tokens(M, wl.LING_TP4.hidden, seed=3_000_000 + seed, device=DEV)
    run_and_check(oracle, layer, host, x, wl.LING_TP4.topk, bias=bias)


def test_all_tokens_on_the_same_experts(oracle, ling):
    """64 tokens forced onto the same 8 experts: 4 groups of 16 per expert."""
    layer, host = ling
    bias = torch.zeros(wl.LING.n_experts)
    forced = [3, 77, 100, 101, 255, 256, 400, 511]
    bias[forced] = 50.0
    x = wl.tokens(64, wl.LING.hidden, seed=42, device=DEV)
    out, idx, st = run_and_check(oracle, layer, host, x, wl.LING.topk, bias=bias)
    assert set(idx.cpu().numpy().ravel().tolist()) == set(forced)
    r = layer.read_routing(64)
    assert r["n_active"] == 8 and r["n_groups"] == 32
    assert np.all(r["grp_cnt"] == 16)
    layer.set_router_bias(None)


def cpu_bucket_sort(idx, E):
    """Reference compaction from the GPU's own routing (integer work)."""
    M, k = idx.shape
    pairs = idx.ravel()
    order = np.argsort(pairs, kind="stable")       # by expert, stable in pair id
    groups = []
    for e in np.unique(pairs):
        pos = np.nonzero(pairs[order] == e)[0]
        for q in range(0, len(pos), 16):
            groups.append((int(e), int(pos[q]), int(min(16, len(pos) - q))))
    return order.astype(np.int32), groups


@pytest.mark.parametrize("M,zipf", [(6, False), (16, True), (64, False), (64, True)])
def test_compaction_matches_cpu_bucket_sort(ling, M, zipf):
    layer, _ = ling
    layer.set_router_bias(wl.zipf_router_bias(wl.LING.n_experts) if zipf else None)
    x = wl.tokens(M, wl.LING.hidden, seed=300 + M, device=DEV)
    tw = torch.empty((M, wl.LING.topk), dtype=torch.float32, device=DEV)
    _, idx = layer(x, topk_w=tw)
    r = layer.read_routing(M)
    idx = idx.cpu().numpy()
    order, groups = cpu_bucket_sort(idx, wl.LING.n_experts)
    assert np.array_equal(r["pair_list"], order)
    assert r["n_active"] == len(np.unique(idx))
    assert r["n_groups"] == len(groups)
    assert [tuple(v) for v in zip(r["grp_expert"], r["grp_start"], r["grp_cnt"])] == groups
    assert np.array_equal(r["pair_w"], tw.cpu().numpy().ravel())
    layer.set_router_bias(None)


def test_pdl_and_graph_are_bitwise_neutral(ling):
    """PDL on/off and graph replay change scheduling only: outputs bit-equal."""
    layer, _ = ling
    layer.set_router_bias(None)
    for M in (6, 1, 16):
        x = wl.tokens(M, wl.LING.hidden, seed=77 + M, device=DEV)
        results = []
        for pdl in (True, False):
            for graph in (False, True, True):  # the second graph call replays
                out, idx = layer(x, pdl=pdl, graph=graph)
                results.append((out.clone(), idx.clone()))
        torch.cuda.synchronize()
        for o, i in results[1:]:
            assert torch.equal(o.view(torch.int16), results[0][0].view(torch.int16))
            assert torch.equal(i, results[0][1])
    # new pointers on a cached graph: the graph is updated, results follow x
    x1 = wl.tokens(6, wl.LING.hidden, seed=1, device=DEV)
    x2 = wl.tokens(6, wl.LING.hidden, seed=2, device=DEV)
    e1, _ = layer(x1)
    e2, _ = layer(x2)
    g1, _ = layer(x1, graph=True)
    g2, _ = layer(x2, graph=True)
    torch.cuda.synchronize()
    assert torch.equal(e1, g1) and torch.equal(e2, g2) and not torch.equal(e1, e2)


def test_graph_capture_by_caller(ling):
    """A caller's CUDA graph of several forward calls replays bit-exactly."""
    layer, _ = ling
    xs = [wl.tokens(6, wl.LING.hidden, seed=500 + i, device=DEV) for i in range(3)]
    outs = [torch.empty_like(x) for x in xs]
    idxs = [torch.empty((6, 8), dtype=torch.int32, device=DEV) for _ in xs]
    ref = [layer(x)[0].clone() for x in xs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for x, o, i in zip(xs, outs, idxs):
                layer(x, out=o, topk_idx=i, stream=s)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, ref):
            assert torch.equal(o, r)


def test_back_to_back_calls_with_changing_M(ling):
    """Calls chained on one stream (PDL, no host synchronisation) while M
    changes from call to call.  Each call reads the partial logits of the
    buffer its parity (odd / even call) picks, which the call before marked
    unwritten for all 64 token rows, so a call with more tokens than the one
    two calls earlier never takes a stale row (16 -> 1 -> 16, 2 -> 64).
    Every result equals the same call made alone."""
    layer, _ = ling
    layer.set_router_bias(None)
    Ms = [16, 1, 16, 6, 64, 2, 64, 1, 6]
    xs = [wl.tokens(M, wl.LING.hidden, seed=900_000 + i, device=DEV) for i, M in enumerate(Ms)]
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


def test_swiglu_epilogue_full_range(oracle, MoELayer):
    """Every finite bf16 gate value through the fused epilogue.

    One-hot tokens make g = W_gate[e][r][pos] and u = W_up[e][r][pos] exactly;
    W_down = [identity; 0] and k = 1 make out[m][r] = h[r] exactly, so the
    output exposes bf16(silu(g) * u) for every (g, u) the layer was given.
    """
    H, E, k, I = 256, 8, 1, 128
    M = 64
    all_g = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    gf = parity.bf16_bits_to_f32(all_g)
    all_g = all_g[np.isfinite(gf)]
    rng = np.random.default_rng(0)
    per_call = M * I
    mism = 0
    subnormal_flush = 0
    total = 0
    bad = []
    for c0 in range(0, all_g.shape[0], per_call):
        gv = all_g[c0:c0 + per_call]
        n = gv.shape[0]
        gate = np.zeros((E, I, H), np.uint16)
        up = np.zeros((E, I, H), np.uint16)
        # |u| < 1 keeps every silu(g) * u finite: an infinite h anywhere in a
        # token's row would turn the identity down projection's 0 * h into NaN
        uvals = wl.bf16_bits(torch.from_numpy(rng.uniform(-0.999, 0.999, n).astype(np.float32))
                             .to(torch.bfloat16))
        # token m uses expert m % E and hidden position m; r = slot within I
        for i in range(n):
            m, r = divmod(i, I)
            gate[m % E, r, m] = gv[i]
            up[m % E, r, m] = uvals[i]
        w_gu = np.concatenate([gate, up], axis=1)
        w_d = np.zeros((E, H, I), np.uint16)
        for e in range(E):
            w_d[e, np.arange(I), np.arange(I)] = 0x3F80       # 1.0
        w_r = np.zeros((E, H), np.uint16)
        for m in range(M):
            w_r[m % E, m] = 0x3F80                            # token m -> expert m % E
        x = np.zeros((M, H), np.uint16)
        x[np.arange(M), np.arange(M)] = 0x3F80
        t = lambda a: wl.bits_to_bf16(a).to(DEV)
        layer = MoELayer(t(w_r), t(w_gu), t(w_d), topk=k)
        out, idx = layer(t(x))
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy().ravel(), np.arange(M) % E)
        got = bits(out.cpu())[:, :I].ravel()[:n]
        for i in range(n):
            g = float(parity.bf16_bits_to_f32(np.array([gv[i]]))[0])
            u = float(parity.bf16_bits_to_f32(np.array([uvals[i]]))[0])
            want = oracle.swiglu_bf16(g, u)
            total += 1
            # the sign of a zero h is not observable through the down
            # projection (1 * -0 + 0 * h' = +0), so zeros compare unsigned
            if got[i] == want or (got[i] & 0x7FFF) == 0 == (want & 0x7FFF):
                continue
            is_sub = (gv[i] & 0x7F80) == 0 and (gv[i] & 0x7F) != 0
            if is_sub and (got[i] & 0x7FFF) == 0:
                subnormal_flush += 1          # a bf16-subnormal gate value read as zero
            elif abs(int(got[i]) - int(want)) <= 1:
                mism += 1                     # one bf16 step (fast exp vs libm exp)
            elif len(bad) < 20:
                bad.append(f"g={g!r} u={u!r}: gpu {got[i]:#06x} oracle {want:#06x}")
            else:
                bad.append("...")
        layer.close()
    assert total == all_g.shape[0]
    assert not bad, f"{len(bad)} epilogue results differ: " + "; ".join(bad[:20])
    assert mism <= 0.001 * total, f"{mism} of {total} differ by one bf16 step"
    # every bf16 subnormal gate value (254 of them) may be read as zero
    assert subnormal_flush <= 254


def test_bad_arguments_on_device(ling):
    from weight_streaming_expert_gb300 import native as N
    layer, _ = ling
    L = N.lib()
    x = wl.tokens(6, wl.LING.hidden, seed=1, device=DEV)
    out = torch.full_like(x, 7.0)
    idx = torch.zeros((6, 8), dtype=torch.int32, device=DEV)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    xp, op, ip = (ctypes.c_void_p(t.data_ptr()) for t in (x, out, idx))
    assert L.moe_forward(layer.handle, ctypes.c_void_p(x.data_ptr() + 2), op, ip, 6, s) == N.MOE_ERR_INVALID_ARG
    assert L.moe_forward(layer.handle, xp, op, ip, 65, s) == N.MOE_ERR_UNSUPPORTED
    assert L.moe_forward(layer.handle, xp, op, ip, -1, s) == N.MOE_ERR_INVALID_ARG
    assert L.moe_forward(layer.handle, xp, op, ip, 0, s) == N.MOE_OK       # no-op
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    assert layer.status() == 0


def test_create_failure_injection_leaks_nothing(MoELayer, monkeypatch):
    from weight_streaming_expert_gb300 import native as N
    w_r, w_gu, w_d = wl.layer_weights(wl.TINY, seed=1)
    w_r, w_gu, w_d = w_r.to(DEV), w_gu.to(DEV), w_d.to(DEV)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for n in (1, 2, 3, 4):
        monkeypatch.setenv("MOE_FAULT_INJECT", f"alloc:{n}")
        with pytest.raises(N.MoEError, match="allocation"):
            MoELayer(w_r, w_gu, w_d, topk=2)
    monkeypatch.delenv("MOE_FAULT_INJECT")
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    layer = MoELayer(w_r, w_gu, w_d, topk=2)   # and a clean create still works
    layer.close()


def test_timed_launch_matches(ling):
    layer, _ = ling
    x = wl.tokens(6, wl.LING.hidden, seed=9, device=DEV)
    ref, ridx = layer(x)
    out = torch.empty_like(x)
    idx = torch.empty_like(ridx)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    layer.forward_timed(x, out, idx, ev)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(idx, ridx)
    assert ev[0].elapsed_time(ev[1]) > 0


# ------------------------------------------------------- layer variants --
# A shared expert every token passes with weight 1, a routed scaling factor
# on every routed weight, and a router bias that picks the experts without
# weighing them (the oracle's moe_forward_ex).

def shared_weights(shape, seed, device="cpu"):
    g = torch.Generator(device=device).manual_seed(seed)
    H, I = shape.hidden, shape.inter
    sgu = (torch.randn(2 * I, H, generator=g, device=device) * wl.WEIGHT_STD).to(torch.bfloat16)
    sd = (torch.randn(H, I, generator=g, device=device) * wl.WEIGHT_STD).to(torch.bfloat16)
    return sgu, sd


def variant_layer(MoELayer, shape, seed, scale, sel_only, device="cpu"):
    w_r, w_gu, w_d = wl.layer_weights(shape, seed=seed, device=device)
    sgu, sd = shared_weights(shape, seed + 1, device=device)
    layer = MoELayer(w_r.to(DEV), w_gu.to(DEV), w_d.to(DEV), topk=shape.topk, shared_gate_up=sgu.to(DEV),
                     shared_down=sd.to(DEV), routed_scale=scale, bias_selection_only=sel_only)
    host = dict(wr=bits(w_r), wgu=bits(w_gu), wd=bits(w_d))
    variant = dict(shared_gate_up=bits(sgu), shared_down=bits(sd), routed_scale=scale,
                   bias_selection_only=sel_only)
    return layer, host, variant


@pytest.mark.parametrize("H,E,k,I,M,scale,sel_only", [
    (256, 16, 2, 128, 1, 1.0, False), (256, 16, 2, 128, 5, 2.5, True), (512, 64, 6, 256, 16, 0.5, True),
    (1280, 40, 3, 256, 23, 2.5, True), (2560, 24, 2, 512, 64, 1.0, False), (1024, 96, 8, 512, 9, 16.0, True)])
def test_variants_small(oracle, MoELayer, H, E, k, I, M, scale, sel_only):
    shape = wl.LayerShape(hidden=H, n_experts=E, topk=k, inter=I)
    layer, host, variant = variant_layer(MoELayer, shape, H + E + k + 77, scale, sel_only)
    bias = torch.from_numpy((np.random.default_rng(E).standard_normal(E) * 0.5).astype(np.float32))
    x = wl.tokens(M, H, seed=M + 500).to(DEV)
    run_and_check(oracle, layer, host, x, k, bias=bias, **variant)
    run_and_check(oracle, layer, host, x, k, bias=None, **variant)
    layer.close()


@pytest.fixture(scope="module")
def ling_variant(MoELayer):
    """Full size, a shared expert, routed scale 2.5, bias for selection only."""
    layer, host, variant = variant_layer(MoELayer, wl.LING, 1200, 2.5, True, device=DEV)
    torch.cuda.empty_cache()
    yield layer, host, variant
    layer.close()


@pytest.mark.parametrize("M,zipf", [(6, False), (1, True), (16, True), (64, False)])
def test_ling_variants(oracle, ling_variant, M, zipf):
    layer, host, variant = ling_variant
    bias = wl.zipf_router_bias(wl.LING.n_experts) if zipf else None
    x = wl.tokens(M, wl.LING.hidden, seed=6_000_000 + M, device=DEV)
    run_and_check(oracle, layer, host, x, wl.LING.topk, bias=bias, **variant)


def test_variant_routing_outputs(oracle, ling_variant):
    """topk_w is the unscaled renormalised weight; the compaction lists the
    shared expert's pairs (id E, weight 1) and the routed pairs scaled."""
    layer, host, variant = ling_variant
    E, k = wl.LING.n_experts, wl.LING.topk
    M = 6
    x = wl.tokens(M, wl.LING.hidden, seed=6_100_000, device=DEV)
    layer.set_router_bias(wl.zipf_router_bias(E))
    tw = torch.empty((M, k), dtype=torch.float32, device=DEV)
    _, idx = layer(x, topk_w=tw)
    r = layer.read_routing(M)
    ref = oracle.moe_forward(bits(x), host["wr"], host["wgu"], host["wd"], k,
                             bias=wl.zipf_router_bias(E).numpy(), **variant)
    same = np.all(idx.cpu().numpy() == ref["idx"], axis=1)
    assert np.allclose(tw.cpu().numpy()[same], ref["w"][same], rtol=1e-5, atol=1e-7)
    pw = r["pair_w"]
    assert np.allclose(pw[:M * k], 2.5 * tw.cpu().numpy().ravel(), rtol=1e-6)
    assert np.all(pw[M * k:] == 1.0)
    shared_groups = r["grp_expert"] == E
    assert shared_groups.sum() == 1 and r["grp_cnt"][shared_groups][0] == M
    assert sorted(r["pair_list"].tolist()) == list(range(M * (k + 1)))
    layer.set_router_bias(None)


# ------------------------------------------------------ fp8 expert weights --
# E4M3 codes with fp32 per-row scales (the oracle's moe_forward_fp8).

def fp8_layer(MoELayer, shape, seed, device="cpu"):
    w_r, q_gu, s_gu, q_d, s_d = wl.fp8_expert_weights(shape, seed=seed, device=device)
    layer = MoELayer.fp8(w_r.to(DEV), q_gu.to(DEV), s_gu.to(DEV), q_d.to(DEV), s_d.to(DEV), topk=shape.topk)
    host = dict(wr=bits(w_r), q_gu=q_gu.cpu().numpy(), s_gu=s_gu.cpu().numpy(), q_d=q_d.cpu().numpy(),
                s_d=s_d.cpu().numpy())
    return layer, host


def run_and_check_fp8(orc, layer, host, x, k, bias=None):
    layer.set_router_bias(bias)
    out, idx = layer(x)
    torch.cuda.synchronize()
    assert layer.status() == 0
    xb = bits(x)
    b = None if bias is None else bias.cpu().numpy()
    return parity.check_against(
        lambda ii: orc.moe_forward_fp8(xb, host["wr"], host["q_gu"], host["s_gu"], host["q_d"], host["s_d"], k,
                                       bias=b, idx_in=ii),
        out.float().cpu().numpy(), idx.cpu().numpy())


@pytest.mark.parametrize("H,E,k,I,M", [(256, 16, 2, 128, 1), (256, 16, 2, 128, 7), (512, 64, 6, 256, 16),
                                       (1280, 40, 3, 256, 23), (2560, 24, 2, 512, 64), (1024, 96, 8, 512, 9)])
def test_fp8_small(oracle, MoELayer, H, E, k, I, M):
    shape = wl.LayerShape(hidden=H, n_experts=E, topk=k, inter=I)
    layer, host = fp8_layer(MoELayer, shape, seed=H + E + k + 99)
    assert layer.info().fp8_experts == 1
    x = wl.tokens(M, H, seed=M + 900).to(DEV)
    run_and_check_fp8(oracle, layer, host, x, k)
    layer.close()


@pytest.fixture(scope="module")
def ling_fp8(MoELayer):
    layer, host = fp8_layer(MoELayer, wl.LING, seed=1300, device=DEV)
    torch.cuda.empty_cache()
    yield layer, host
    layer.close()


@pytest.mark.parametrize("M,zipf", [(6, False), (1, False), (16, True), (64, False)])
def test_ling_fp8(oracle, ling_fp8, M, zipf):
    layer, host = ling_fp8
    bias = wl.zipf_router_bias(wl.LING.n_experts) if zipf else None
    x = wl.tokens(M, wl.LING.hidden, seed=7_000_000 + M, device=DEV)
    run_and_check_fp8(oracle, layer, host, x, wl.LING.topk, bias=bias)
