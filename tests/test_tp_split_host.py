"""CPU tests of the tensor-parallel split's host side (no GPU).

The post's deployment splits every expert's intermediate rows over 4 GPUs
and ends the MoE chain with an all-reduce of the partial outputs ("PDL: the
latency floor of stacked small kernels").  Here:
  * tp_slice picks the right rows: the oracle run on the G slices gives fp32
    partial combines that sum to the oracle's unsplit combine (the down
    projection is a sum over the intermediate rows, so it splits exactly up
    to fp32 summation order), and a slice whose gate and up rows do not
    belong together breaks that;
  * the exchange step as bench.py runs it (an all-gather of the fp32 parts,
    then their ordered sum and one bf16 rounding) on two gloo ranks gives the
    same bits on both ranks, and the unsplit layer's output under the usual
    parity rule.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from tests import parity
from weight_streaming_expert_gb300 import workloads as wl
from weight_streaming_expert_gb300.layer import tp_slice

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bits(t):
    return wl.bf16_bits(t)


def slice_accs(oracle, x, w_r, w_gu, w_d, k, G, idx_in=None):
    accs = []
    for r in range(G):
        gu, d = tp_slice(w_gu, w_d, r, G)
        accs.append(oracle.moe_forward(bits(x), bits(w_r), bits(gu), bits(d), k, idx_in=idx_in)["acc"])
    return accs


@pytest.mark.parametrize("H,E,k,I,G,M", [(256, 16, 2, 256, 2, 3), (512, 24, 4, 512, 4, 5), (256, 8, 1, 512, 4, 1)])
def test_oracle_slices_sum_to_the_unsplit_layer(oracle, H, E, k, I, G, M):
    shape = wl.LayerShape(hidden=H, n_experts=E, topk=k, inter=I)
    w_r, w_gu, w_d = wl.layer_weights(shape, seed=H + E + G)
    x = wl.tokens(M, H, seed=G)
    full = oracle.moe_forward(bits(x), bits(w_r), bits(w_gu), bits(w_d), k)
    accs = slice_accs(oracle, x, w_r, w_gu, w_d, k, G)
    total = accs[0].astype(np.float64)
    for a in accs[1:]:
        total += a
    scale = np.abs(full["acc"]).max()
    assert np.abs(total - full["acc"]).max() <= 1e-5 * scale + 1e-7
    # gate rows of one slice with up rows of another: not the layer any more
    gu0, d0 = tp_slice(w_gu, w_d, 0, G)
    gu1, _ = tp_slice(w_gu, w_d, 1, G)
    s = I // G
    mixed = torch.cat([gu0[:, :s], gu1[:, s:]], dim=1).contiguous()
    bad = oracle.moe_forward(bits(x), bits(w_r), bits(mixed), bits(d0), k)["acc"]
    assert np.abs(bad - accs[0]).max() > 1e-3 * scale


def test_tp_slice_shapes_and_rows():
    w_gu = torch.arange(2 * 8 * 4, dtype=torch.float32).view(2, 8, 4)   # E 2, I 4, H 4
    w_d = torch.arange(2 * 4 * 4, dtype=torch.float32).view(2, 4, 4)
    gu, d = tp_slice(w_gu, w_d, 1, 2)
    assert gu.shape == (2, 4, 4) and d.shape == (2, 4, 2)
    assert torch.equal(gu[:, :2], w_gu[:, 2:4]) and torch.equal(gu[:, 2:], w_gu[:, 6:8])
    assert torch.equal(d, w_d[:, :, 2:4])
    with pytest.raises(ValueError):
        tp_slice(w_gu, w_d, 0, 3)


WORKER = r"""
import os, sys, hashlib
sys.path.insert(0, {root!r})
import numpy as np, torch
import bench
from oracle.oracle import Oracle
from tests import parity
from weight_streaming_expert_gb300 import workloads as wl
from weight_streaming_expert_gb300.layer import tp_slice
rank, ws, local, pg = bench.dist_setup(2)
assert ws == 2 and pg is not None
orc = Oracle()
shape = wl.LayerShape(hidden=512, n_experts=24, topk=4, inter=256)
w_r, w_gu, w_d = wl.layer_weights(shape, seed=77)
x = wl.tokens(6, 512, seed=78)
b = wl.bf16_bits
gu, d = tp_slice(w_gu, w_d, rank, ws)
part = torch.from_numpy(orc.moe_forward(b(x), b(w_r), b(gu), b(d), shape.topk)["acc"])
parts = bench.tp_exchange(part, pg, ws)              # [2, M, H], the same on both ranks
assert tuple(parts.shape) == (2, 6, 512)
assert torch.equal(parts[rank], part)
s = parts[0].clone()
for p in range(1, ws):
    s = s + parts[p]                                  # fp32, in rank order
out = s.to(torch.bfloat16)                            # one rounding
st = parity.check_layer(orc, b(x), b(w_r), b(w_gu), b(w_d), shape.topk, out.float().numpy(),
                        orc.moe_forward(b(x), b(w_r), b(gu), b(d), shape.topk)["idx"])
print("ok", rank, hashlib.sha256(b(out).tobytes()).hexdigest()[:16], flush=True)
pg.destroy_process_group()
"""


def test_two_rank_exchange_gloo(tmp_path):
    script = tmp_path / "tp.py"
    script.write_text(WORKER.format(root=ROOT))
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                        "--master-addr=127.0.0.1", "--master-port=29547", str(script)],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l.split() for l in r.stdout.splitlines() if l.startswith("ok")]
    assert len(lines) == 2
    assert lines[0][2] == lines[1][2], "the ranks' combined outputs differ"
