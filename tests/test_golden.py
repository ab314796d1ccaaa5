"""The oracle built on this host reproduces the committed oracle record."""
import os

import numpy as np

from weight_streaming_expert_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_seed0.txt")


def load_tiny_golden():
    recs, cur = {}, None
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        if key == "M":
            cur = int(vals[0])
            recs[cur] = {}
        elif key == "idx":
            recs[cur]["idx"] = np.array([int(v) for v in vals], np.int32)
        elif key == "w":
            recs[cur]["w"] = np.array([int(v, 16) for v in vals], np.uint32).view(np.float32)
        elif key == "out":
            recs[cur]["out"] = np.array([int(v, 16) for v in vals], np.uint16)
    return recs


def test_oracle_matches_committed_record(oracle):
    recs = load_tiny_golden()
    assert set(recs) == {1, 4}
    for M, rec in recs.items():
        w_r, w_gu, w_d, x = wl.tiny_case(M=M, seed=0)
        res = oracle.moe_forward(wl.bf16_bits(x), wl.bf16_bits(w_r), wl.bf16_bits(w_gu),
                                 wl.bf16_bits(w_d), wl.TINY.topk)
        assert np.array_equal(res["idx"].ravel(), rec["idx"])
        assert np.allclose(res["w"].ravel(), rec["w"], rtol=3e-7, atol=0)
        # libm exp may differ by an ulp across hosts: allow one bf16 step
        d = np.abs(res["out"].ravel().astype(np.int64) - rec["out"].astype(np.int64))
        assert d.max() <= 1 and np.mean(d == 0) > 0.99


def test_oracle_lm_head_matches_committed_record(oracle):
    path = os.path.join(os.path.dirname(GOLDEN), "lm_head_seed21.txt")
    vals = [l for l in open(path) if not l.startswith("#") and l.strip()][0].split()
    want = np.array([int(v, 16) for v in vals], np.uint32).view(np.float32).reshape(2, 333)
    got = oracle.lm_head(wl.bf16_bits(wl.tokens(2, 256, seed=22)), wl.bf16_bits(wl.lm_head_weight(333, 256, seed=21)))
    # fp32 sums in a fixed order, no transcendental: the same on every host
    assert np.array_equal(got, want)
