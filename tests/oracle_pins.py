"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``Oracle`` and raises AssertionError when the
oracle disagrees with an independent fact:
  * library routines (torch's fp32->bf16 rounding, numpy sorting),
  * a float64 dense brute force that evaluates EVERY expert and then masks
    with a dense routing vector (a different algorithm from the oracle's
    sparse loop),
  * closed forms (one-hot routing = one dense SwiGLU MLP; zero input;
    uniform logits give w = 1/k),
  * invariants (sum of routing weights = 1; expert relabelling; identical
    tokens give identical rows).
``tests/test_oracle_pins.py`` runs them against the real oracle and, to show
they have teeth, against copies of the oracle with a planted mistake.
"""
from __future__ import annotations

import numpy as np
import torch

from weight_streaming_expert_gb300 import workloads as wl


# ----------------------------------------------------------------- helpers --

def f32_of_bits(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round_torch(a):
    """Library rounding fp32 -> bf16 (torch), returned as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def silu64(g):
    return g / (1.0 + np.exp(-g))


def dense_reference(x, w_r, w_gu, w_d, k, bias=None):
    """float64 brute force over ALL experts, then a dense routing mask.

    Returns (idx [M,k] by float64 logits, acc [M,H] float64 before the cast).
    h is rounded to bf16 (library rounding) like the layer does; everything
    else stays float64.
    """
    X = f32_of_bits(x).astype(np.float64)             # [M,H]
    Wr = f32_of_bits(w_r).astype(np.float64)          # [E,H]
    Wgu = f32_of_bits(w_gu).astype(np.float64)        # [E,2I,H]
    Wd = f32_of_bits(w_d).astype(np.float64)          # [E,H,I]
    E, twoI, H = Wgu.shape
    I = twoI // 2
    logits = X @ Wr.T
    if bias is not None:
        logits = logits + np.asarray(bias, np.float64)[None, :]
    M = X.shape[0]
    # every expert on every token
    G = np.einsum("eih,mh->mei", Wgu[:, :I, :], X)    # [M,E,I]
    U = np.einsum("eih,mh->mei", Wgu[:, I:, :], X)
    hh = silu64(G) * U
    hh = f32_of_bits(bf16_round_torch(hh.astype(np.float32))).astype(np.float64)
    Y = np.einsum("ehi,mei->meh", Wd, hh)             # [M,E,H]
    # dense routing vector: softmax over all experts, zero outside the top-k,
    # renormalised over the kept entries
    dense = np.zeros((M, E))
    idx = np.zeros((M, k), np.int64)
    for m in range(M):
        order = np.lexsort((np.arange(E), -logits[m]))  # by logit desc, then id asc
        idx[m] = order[:k]
        p = np.exp(logits[m] - logits[m].max())
        p /= p.sum()
        mask = np.zeros(E, bool)
        mask[order[:k]] = True
        dense[m] = np.where(mask, p, 0.0)
        dense[m] /= dense[m].sum()
    acc = np.einsum("me,meh->mh", dense, Y)
    return idx, acc, logits


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _np(t):
    return wl.bf16_bits(t)


def tiny(M=3, seed=0, shape=wl.TINY):
    w_r, w_gu, w_d, x = wl.tiny_case(M=M, seed=seed, shape=shape)
    return _np(x), _np(w_r), _np(w_gu), _np(w_d)


# -------------------------------------------------------------------- pins --

def pin_bf16_rounding(orc):
    # hand cases: exact, ties to even (down and up), negative, carry into exponent
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,          # tie between 0x3F80 and 0x3F81 -> even 0x3F80
        1.0 + 3 * 2.0 ** -8: 0x3F82,      # tie between 0x3F81 and 0x3F82 -> even 0x3F82
        1.0 + 2.0 ** -8 + 2.0 ** -20: 0x3F81,  # just above the tie -> up
        -1.5: 0xBFC0,
        2.0 - 2.0 ** -9: 0x4000,          # rounds up across the exponent boundary
        0.0: 0x0000,
    }
    for f, want in cases.items():
        got = orc.f32_to_bf16(f)
        assert got == want, f"bf16({f!r}) = {got:#06x}, want {want:#06x}"
    # library routine on many values
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 3,
                           rng.standard_normal(1000).astype(np.float32) * 1e-3])
    lib = bf16_round_torch(vals)
    got = np.array([orc.f32_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, lib), "fp32->bf16 disagrees with torch rounding"
    # bf16 -> fp32 is exact
    for b in (0x3F80, 0xBFC0, 0x0001, 0x7F7F, 0x4049):
        want = float(f32_of_bits(np.array([b], np.uint16))[0])
        assert orc.bf16_to_f32(b) == want


def pin_router_logits(orc):
    x, w_r, _, _ = tiny(M=4, seed=3)
    lg = orc.router_logits(x, w_r)
    X = f32_of_bits(x).astype(np.float64)
    Wr = f32_of_bits(w_r).astype(np.float64)
    ref = X @ Wr.T
    bound = 1e-5 * (np.abs(X) @ np.abs(Wr).T) + 1e-6
    assert lg.shape == ref.shape
    assert np.all(np.abs(lg - ref) <= bound), "router logits != float64 matmul"
    b = np.linspace(-2, 2, w_r.shape[0]).astype(np.float32)
    lgb = orc.router_logits(x, w_r, bias=b)
    assert np.all(np.abs(lgb - (ref + b[None, :])) <= bound + 1e-6), "bias not added"


def pin_topk_brute_force(orc):
    rng = np.random.default_rng(5)
    for E, k in ((16, 2), (16, 1), (40, 8), (512, 8), (7, 7)):
        lg = rng.standard_normal((6, E)).astype(np.float32)
        # plant exact ties, including across the k boundary
        lg[0, 3] = lg[0, 5] = lg[0].max() + 1.0
        lg[1, :] = 0.5
        lg[2, E - 1] = lg[2, 0] = lg[2].max() + 0.25
        idx, w = orc.topk_softmax(lg, k)
        for m in range(lg.shape[0]):
            order = np.lexsort((np.arange(E), -lg[m].astype(np.float64)))
            assert list(idx[m]) == list(order[:k]), f"top-k mismatch E={E} k={k} m={m}"
            p = np.exp(lg[m].astype(np.float64) - lg[m].max())
            p /= p.sum()
            ref = p[order[:k]] / p[order[:k]].sum()
            assert np.allclose(w[m], ref, rtol=2e-6, atol=1e-7), "renormalised softmax weights"
            assert abs(float(w[m].astype(np.float64).sum()) - 1.0) < 1e-6, "weights must sum to 1"
        # weights for a given set equal the oracle's own weights on its own set
        for m in range(lg.shape[0]):
            ws = orc.weights_for_set(lg[m], idx[m])
            assert np.allclose(ws, w[m], rtol=1e-6, atol=1e-8)


def pin_swiglu(orc):
    # closed forms
    assert orc.swiglu_bf16(0.0, 3.0) == 0x0000
    assert orc.swiglu_bf16(2.0, 0.0) == 0x0000
    assert orc.swiglu_bf16(30.0, 1.0) == orc.f32_to_bf16(30.0)      # silu(x) -> x for large x
    assert f32_of_bits(np.array([orc.swiglu_bf16(-30.0, 1.0)], np.uint16))[0] <= 0.0
    assert abs(float(f32_of_bits(np.array([orc.swiglu_bf16(-30.0, 1.0)], np.uint16))[0])) < 1e-10
    # full range of finite bf16 gate values, one rounding on the product
    g_bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    g = f32_of_bits(g_bits)
    fin = np.isfinite(g) & (np.abs(g) < 80.0)
    g = g[fin][::3]
    rng = np.random.default_rng(11)
    u = rng.standard_normal(g.shape[0]).astype(np.float32)
    ref = bf16_round_torch((silu64(g.astype(np.float64)) * u.astype(np.float64)).astype(np.float32))
    got = np.array([orc.swiglu_bf16(float(a), float(b)) for a, b in zip(g, u)], np.uint16)
    same = float(np.mean(got == ref))
    # the float64 reference and the fp32 formula round to the same bf16
    # except within an fp32 ulp of a rounding boundary
    assert same > 0.999, f"silu*u single rounding matches on only {same:.4f}"
    diff_ulp = np.abs(got.astype(np.int64) - ref.astype(np.int64))
    assert diff_ulp.max() <= 1


def pin_dense_bruteforce(orc):
    for (M, seed, shape) in ((1, 0, wl.TINY), (3, 1, wl.TINY),
                             (4, 2, wl.LayerShape(hidden=64, n_experts=12, topk=4, inter=32)),
                             (5, 3, wl.LayerShape(hidden=32, n_experts=8, topk=1, inter=16))):
        x, w_r, w_gu, w_d = tiny(M=M, seed=seed, shape=shape)
        k = shape.topk
        res = orc.moe_forward(x, w_r, w_gu, w_d, k)
        idx64, acc64, lg64 = dense_reference(x, w_r, w_gu, w_d, k)
        assert np.array_equal(res["idx"], idx64), "routing differs from float64 brute force"
        assert rel_l2(res["acc"], acc64) < 2e-3, f"oracle vs dense brute force rel-L2 {rel_l2(res['acc'], acc64)}"
        assert np.max(np.abs(res["acc"] - acc64)) < 2e-3
        # final cast is one RNE rounding of acc
        assert np.array_equal(res["out"], bf16_round_torch(res["acc"]))
    # with a router bias (skewed routing)
    shape = wl.TINY
    x, w_r, w_gu, w_d = tiny(M=3, seed=9)
    b = wl.zipf_router_bias(shape.n_experts).numpy()
    res = orc.moe_forward(x, w_r, w_gu, w_d, shape.topk, bias=b)
    idx64, acc64, _ = dense_reference(x, w_r, w_gu, w_d, shape.topk, bias=b)
    assert np.array_equal(res["idx"], idx64), "biased routing differs from brute force"
    assert rel_l2(res["acc"], acc64) < 2e-3


def pin_one_hot_router(orc):
    """One expert forced (bias +1e4), k = 1: the layer is one dense SwiGLU MLP."""
    shape = wl.TINY
    x, w_r, w_gu, w_d = tiny(M=3, seed=4)
    E, I = shape.n_experts, shape.inter
    for e_star in (0, 7, E - 1):
        b = np.zeros(E, np.float32)
        b[e_star] = 1e4
        res = orc.moe_forward(x, w_r, w_gu, w_d, 1, bias=b)
        assert np.all(res["idx"] == e_star)
        assert np.all(res["w"] == 1.0)
        X = f32_of_bits(x).astype(np.float64)
        Wg = f32_of_bits(w_gu[e_star, :I]).astype(np.float64)
        Wu = f32_of_bits(w_gu[e_star, I:]).astype(np.float64)
        Wd = f32_of_bits(w_d[e_star]).astype(np.float64)
        hh = silu64(X @ Wg.T) * (X @ Wu.T)
        hh = f32_of_bits(bf16_round_torch(hh.astype(np.float32))).astype(np.float64)
        mlp = hh @ Wd.T
        assert rel_l2(res["acc"], mlp) < 2e-3, "one-hot routing != dense SwiGLU MLP"


def pin_special_cases(orc):
    shape = wl.TINY
    x, w_r, w_gu, w_d = tiny(M=2, seed=6)
    k = 4
    # x = 0: zero logits (all tied) -> experts 0..k-1 with w = 1/k; out = 0 exactly
    z = np.zeros_like(x)
    res = orc.moe_forward(z, w_r, w_gu, w_d, k)
    assert np.all(res["out"] == 0)
    assert np.all(res["idx"] == np.arange(k)[None, :])
    assert np.all(res["w"] == np.float32(1.0 / k))
    # W_r = 0: same routing, nonzero output equal to the uniform mix of experts 0..k-1
    res0 = orc.moe_forward(x, np.zeros_like(w_r), w_gu, w_d, k)
    assert np.all(res0["idx"] == np.arange(k)[None, :])
    assert np.all(res0["w"] == np.float32(1.0 / k))
    # identical tokens -> identical rows
    xx = np.repeat(x[:1], 3, axis=0)
    r2 = orc.moe_forward(xx, w_r, w_gu, w_d, shape.topk)
    assert np.array_equal(r2["out"][0], r2["out"][1]) and np.array_equal(r2["out"][0], r2["out"][2])


def pin_expert_permutation(orc):
    shape = wl.TINY
    x, w_r, w_gu, w_d = tiny(M=3, seed=8)
    E = shape.n_experts
    perm = np.random.default_rng(2).permutation(E)       # new expert i is old expert perm[i]
    inv = np.argsort(perm)
    a = orc.moe_forward(x, w_r, w_gu, w_d, shape.topk)
    b = orc.moe_forward(x, w_r[perm], w_gu[perm], w_d[perm], shape.topk)
    assert np.array_equal(inv[a["idx"]], b["idx"]), "indices must map through the permutation"
    assert np.allclose(a["acc"], b["acc"], rtol=1e-6, atol=1e-7)


def pin_lm_head(orc):
    """The vocabulary projection against a float64 matmul (ragged vocabulary),
    a one-hot token (one exact product per logit) and a zero token."""
    H, V = 256, 333
    w = _np(wl.lm_head_weight(V, H, seed=21))
    x = _np(wl.tokens(3, H, seed=22))
    lg = orc.lm_head(x, w)
    X = f32_of_bits(x).astype(np.float64)
    W = f32_of_bits(w).astype(np.float64)
    ref = X @ W.T
    bound = 1e-5 * (np.abs(X) @ np.abs(W).T) + 1e-6
    assert lg.shape == (3, V)
    assert np.all(np.abs(lg - ref) <= bound), "lm_head != float64 matmul"
    c = 0x3FC0                                # bf16 1.5
    oh = np.zeros((2, H), np.uint16)
    oh[0, 7] = c
    oh[1, H - 1] = c
    lo = orc.lm_head(oh, w)
    assert np.array_equal(lo[0], (1.5 * W[:, 7]).astype(np.float32)), "one-hot token: column 7"
    assert np.array_equal(lo[1], (1.5 * W[:, H - 1]).astype(np.float32)), "one-hot token: last column"
    assert not np.any(orc.lm_head(np.zeros((1, H), np.uint16), w)), "zero token"


def _shared_weights(shape, seed):
    g = torch.Generator().manual_seed(seed)
    H, I = shape.hidden, shape.inter
    sgu = (torch.randn(2 * I, H, generator=g) * wl.WEIGHT_STD).to(torch.bfloat16)
    sd = (torch.randn(H, I, generator=g) * wl.WEIGHT_STD).to(torch.bfloat16)
    return _np(sgu), _np(sd)


def _dense_mlp(x, w_gu, w_d):
    """float64 SwiGLU MLP with h rounded to bf16 (library rounding)."""
    I = w_d.shape[1]
    X = f32_of_bits(x).astype(np.float64)
    Wg = f32_of_bits(w_gu[:I]).astype(np.float64)
    Wu = f32_of_bits(w_gu[I:]).astype(np.float64)
    Wd = f32_of_bits(w_d).astype(np.float64)
    hh = silu64(X @ Wg.T) * (X @ Wu.T)
    hh = f32_of_bits(bf16_round_torch(hh.astype(np.float32))).astype(np.float64)
    return hh @ Wd.T


def pin_shared_expert_and_scale(orc):
    """Shared expert + routed scale against the dense brute force: acc =
    scale * (routed mixture) + shared MLP; scale 0 leaves the shared MLP
    alone; no shared expert and scale 1 is the plain layer, bit for bit."""
    shape = wl.TINY
    x, w_r, w_gu, w_d = tiny(M=4, seed=12)
    sgu, sd = _shared_weights(shape, 13)
    shared = _dense_mlp(x, sgu, sd)
    _, routed, _ = dense_reference(x, w_r, w_gu, w_d, shape.topk)
    for scale in (0.0, 1.0, 2.5):
        r = orc.moe_forward(x, w_r, w_gu, w_d, shape.topk, shared_gate_up=sgu, shared_down=sd, routed_scale=scale)
        assert rel_l2(r["acc"], scale * routed + shared) < 2e-3, f"shared + {scale} x routed != dense brute force"
    r0 = orc.moe_forward(x, w_r, w_gu, w_d, shape.topk, shared_gate_up=sgu, shared_down=sd, routed_scale=0.0)
    assert rel_l2(r0["acc"], shared) < 2e-3, "scale 0: the shared expert alone"
    plain = orc.moe_forward(x, w_r, w_gu, w_d, shape.topk)
    same = orc.moe_forward(x, w_r, w_gu, w_d, shape.topk, routed_scale=1.0)
    assert np.array_equal(plain["out"], same["out"]) and np.array_equal(plain["acc"], same["acc"])


def pin_selection_only_bias(orc):
    """The bias picks the experts, the unbiased softmax weighs them (numpy
    lexsort and a float64 softmax over the chosen set)."""
    shape = wl.TINY
    x, w_r, w_gu, w_d = tiny(M=5, seed=14)
    E, k = shape.n_experts, shape.topk
    b = (np.random.default_rng(15).standard_normal(E) * 0.5).astype(np.float32)
    r = orc.moe_forward(x, w_r, w_gu, w_d, k, bias=b, bias_selection_only=True)
    X = f32_of_bits(x).astype(np.float64)
    Wr = f32_of_bits(w_r).astype(np.float64)
    lg = X @ Wr.T
    moved = 0
    for m in range(x.shape[0]):
        sel = lg[m] + b
        order = np.lexsort((np.arange(E), -sel))[:k]
        assert np.array_equal(r["idx"][m], order), "selection must follow the biased logits"
        p = np.exp(lg[m][order] - lg[m][order].max())
        assert np.allclose(r["w"][m], p / p.sum(), rtol=1e-5, atol=1e-7), "weights: unbiased softmax over the set"
        moved += not np.array_equal(order, np.lexsort((np.arange(E), -lg[m]))[:k])
    assert moved > 0, "the bias must change some token's selection in this case"
    rb = orc.moe_forward(x, w_r, w_gu, w_d, k, bias=b)
    assert not np.allclose(rb["w"], r["w"]), "the two bias modes must weigh differently"


def pin_e4m3_decode(orc):
    """Every E4M3 code against torch's float8_e4m3fn, plus hand values."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).float().numpy()
    got = np.array([orc.e4m3_to_f32(c) for c in range(256)], np.float32)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2, "NaN codes are S.1111.111 only"
    assert np.array_equal(got[~nan], lib[~nan]), "E4M3 decode != torch"
    for code, val in ((0x7E, 448.0), (0x38, 1.0), (0x01, 2.0 ** -9), (0xC6, -3.5), (0x08, 2.0 ** -6)):
        assert orc.e4m3_to_f32(code) == val


def _fp8_tiny(seed):
    shape = wl.TINY
    w_r, q_gu, s_gu, q_d, s_d = wl.fp8_expert_weights(shape, seed=seed)
    x = wl.tokens(4, shape.hidden, seed=seed + 1)
    return shape, _np(x), _np(w_r), q_gu.numpy(), s_gu.numpy(), q_d.numpy(), s_d.numpy()


def pin_fp8_unit_scales_are_bf16(orc):
    """With unit scales the fp8 layer is the bf16 layer on the decoded codes
    (every E4M3 value is a bf16 value), bit for bit."""
    shape, x, w_r, q_gu, _, q_d, _ = _fp8_tiny(31)
    E, I, H = shape.n_experts, shape.inter, shape.hidden
    one_gu, one_d = np.ones((E, 2 * I), np.float32), np.ones((E, H), np.float32)
    f8 = orc.moe_forward_fp8(x, w_r, q_gu, one_gu, q_d, one_d, shape.topk)
    dec = lambda q: bf16_round_torch(torch.from_numpy(q).view(torch.float8_e4m3fn).float().numpy())
    bf = orc.moe_forward(x, w_r, dec(q_gu), dec(q_d), shape.topk)
    assert np.array_equal(f8["idx"], bf["idx"])
    assert np.array_equal(f8["acc"], bf["acc"]) and np.array_equal(f8["out"], bf["out"])


def pin_fp8_dense(orc):
    """Per-row scales against a float64 dense brute force on the dequantized
    weights diag(scale) * decode(codes)."""
    shape, x, w_r, q_gu, s_gu, q_d, s_d = _fp8_tiny(33)
    I = shape.inter
    f8 = orc.moe_forward_fp8(x, w_r, q_gu, s_gu, q_d, s_d, shape.topk)
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    Wgu = dec(q_gu) * s_gu[:, :, None].astype(np.float64)
    Wd = dec(q_d) * s_d[:, :, None].astype(np.float64)
    X = f32_of_bits(x).astype(np.float64)
    Wr = f32_of_bits(w_r).astype(np.float64)
    logits = X @ Wr.T
    G = np.einsum("eih,mh->mei", Wgu[:, :I, :], X)
    U = np.einsum("eih,mh->mei", Wgu[:, I:, :], X)
    hh = f32_of_bits(bf16_round_torch((silu64(G) * U).astype(np.float32))).astype(np.float64)
    Y = np.einsum("ehi,mei->meh", Wd, hh)
    M, E = X.shape[0], shape.n_experts
    acc = np.zeros((M, shape.hidden))
    for m in range(M):
        order = np.lexsort((np.arange(E), -logits[m]))[:shape.topk]
        assert np.array_equal(f8["idx"][m], order)
        p = np.exp(logits[m][order] - logits[m][order].max())
        acc[m] = (p / p.sum()) @ Y[m, order]
    assert rel_l2(f8["acc"], acc) < 2e-3, "fp8 layer != dense brute force on dequantized weights"


ALL_PINS = [pin_bf16_rounding, pin_router_logits, pin_topk_brute_force, pin_swiglu,
            pin_dense_bruteforce, pin_one_hot_router, pin_special_cases, pin_expert_permutation,
            pin_lm_head, pin_shared_expert_and_scale, pin_selection_only_bias, pin_e4m3_decode,
            pin_fp8_unit_scales_are_bf16, pin_fp8_dense]
