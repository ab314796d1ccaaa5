"""Writes tests/golden/tiny_seed0.txt and lm_head_seed21.txt from the CPU oracle.

The fixture is a regression record of the oracle on the small oracle-check
layer (hidden 256, 16 experts, top-2, inter 128, all tensors from seed 0),
for M = 1 and M = 4.  It lets a run on another host (the GPU machine is an
Arm host) confirm that the oracle it builds there computes what the pinned
oracle computed here.  Only the oracle and the seeded input generator are
called.  lm_head_seed21.txt does the same for the vocabulary projection
(hidden 256, a ragged vocabulary of 333 rows from seed 21, two tokens from
seed 22).

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle.oracle import Oracle  # noqa: E402
from weight_streaming_expert_gb300 import workloads as wl  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_seed0.txt")
OUT_LM = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lm_head_seed21.txt")


def main():
    orc = Oracle()
    lines = ["# oracle output on the small oracle-check layer, seed 0 (see make_golden.py)",
             "# M  idx[M*k]  w[M*k] (fp32 hex)  out[M*H] (bf16 hex)"]
    for M in (1, 4):
        w_r, w_gu, w_d, x = wl.tiny_case(M=M, seed=0)
        res = orc.moe_forward(wl.bf16_bits(x), wl.bf16_bits(w_r), wl.bf16_bits(w_gu),
                              wl.bf16_bits(w_d), wl.TINY.topk)
        lines.append(f"M {M}")
        lines.append("idx " + " ".join(str(int(v)) for v in res["idx"].ravel()))
        lines.append("w " + " ".join(f"{int(v):08x}" for v in res["w"].ravel().view(np.uint32)))
        lines.append("out " + " ".join(f"{int(v):04x}" for v in res["out"].ravel()))
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print("wrote", OUT)
    w = wl.bf16_bits(wl.lm_head_weight(333, 256, seed=21))
    x = wl.bf16_bits(wl.tokens(2, 256, seed=22))
    lg = orc.lm_head(x, w)
    with open(OUT_LM, "w") as f:
        f.write("# oracle lm_head logits, hidden 256, vocab 333 (seed 21), 2 tokens (seed 22); fp32 hex, row-major\n")
        f.write(" ".join(f"{int(v):08x}" for v in lg.ravel().view(np.uint32)) + "\n")
    print("wrote", OUT_LM)


if __name__ == "__main__":
    main()
