"""GPU-vs-oracle acceptance rule shared by the GPU tests, smoke and bench.

Routing: the GPU's experts of a token must equal the oracle's, in order,
except where the oracle's logits at the disagreement are a near-tie:
|a - b| <= TIE_REL * max(|a|, |b|) + TIE_ABS.  At a near-tie the GPU's own
set is scored with the oracle's weights for that set (the oracle is re-run
with the GPU's indices) and the outputs are compared against that.

Outputs: max |gpu - oracle| <= 2e-2 and ||gpu - oracle|| / ||oracle|| <= 1e-2,
on the bf16 outputs read as fp32.
"""
from __future__ import annotations

import numpy as np

TIE_REL = 1e-3
TIE_ABS = 1e-5        # logits near 0: fp32 summation-order noise of a 2560-term dot
MAX_ABS = 2e-2
MAX_REL_L2 = 1e-2


def bf16_bits_to_f32(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def near(a, b):
    return abs(a - b) <= TIE_REL * max(abs(a), abs(b)) + TIE_ABS


def routing_ok(gpu_idx_row, ora_idx_row, logits_row):
    """True if the GPU's ordered top-k is the oracle's, up to near-ties."""
    g = list(gpu_idx_row)
    o = list(ora_idx_row)
    if g == o:
        return True
    k = len(o)
    if len(set(g)) != k or min(g) < 0 or max(g) >= logits_row.shape[0]:
        return False
    l = logits_row.astype(np.float64)
    kth = l[o[-1]]
    # every chosen expert must be at least the oracle's k-th logit (up to a tie),
    # every expert left out at most it (up to a tie)
    chosen = set(g)
    for e in g:
        if l[e] < kth and not near(l[e], kth):
            return False
    for e in o:
        if e not in chosen and not near(l[e], kth):
            return False
    # order: non-increasing oracle logits up to ties
    for a_, b_ in zip(g[:-1], g[1:]):
        if l[a_] < l[b_] and not near(l[a_], l[b_]):
            return False
    return True


def compare_outputs(gpu_out_f32, ora_out_bits):
    want = bf16_bits_to_f32(ora_out_bits).astype(np.float64)
    got = np.asarray(gpu_out_f32, np.float64)
    err = np.abs(got - want)
    max_abs = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)) if err.size else 0.0
    return max_abs, rel


def check_against(ref_fn, gpu_out_f32, gpu_idx, max_abs=MAX_ABS, max_rel=MAX_REL_L2):
    """The acceptance rule against any oracle layer: ref_fn(idx_in) returns the
    oracle's dict (out, idx, logits, ...) with its own routing (idx_in None) or
    scored on the GPU's experts.  Returns stats; raises AssertionError."""
    ref = ref_fn(None)
    gpu_idx = np.asarray(gpu_idx, np.int32)
    ties = 0
    for m in range(gpu_idx.shape[0]):
        if not np.array_equal(gpu_idx[m], ref["idx"][m]):
            assert routing_ok(gpu_idx[m], ref["idx"][m], ref["logits"][m]), (
                f"token {m}: gpu experts {gpu_idx[m].tolist()} vs oracle {ref['idx'][m].tolist()} "
                f"is not a near-tie")
            ties += 1
    if ties:
        ref = ref_fn(gpu_idx)
    max_abs_err, rel = compare_outputs(gpu_out_f32, ref["out"])
    assert max_abs_err <= max_abs and rel <= max_rel, (
        f"outputs: max-abs {max_abs_err:.3e} (<= {max_abs}) rel-L2 {rel:.3e} (<= {max_rel})")
    return dict(near_tie_tokens=ties, max_abs=max_abs_err, rel_l2=rel, ref=ref)


def check_layer(orc, x_bits, wr_bits, wgu_bits, wd_bits, k, gpu_out_f32, gpu_idx, bias=None,
                max_abs=MAX_ABS, max_rel=MAX_REL_L2, **variant):
    """Full acceptance check; returns a dict of stats, raises AssertionError on failure.
    ``variant``: the oracle's layer-variant arguments (shared_gate_up,
    shared_down, routed_scale, bias_selection_only)."""
    return check_against(lambda ii: orc.moe_forward(x_bits, wr_bits, wgu_bits, wd_bits, k, bias=bias, idx_in=ii,
                                                    **variant),
                         gpu_out_f32, gpu_idx, max_abs, max_rel)
