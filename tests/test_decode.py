"""Split-KV decoding (fa_decode_splitkv + fa_splitkv_merge) against the fp64
oracle: the merged output against full single-query attention, and the
phase-1 partials against the oracle's own partials (uneven and empty
partitions included)."""
import math

import numpy as np
import pytest
import torch

import exact_attention_54_gb300 as fa
import oracle
from exact_attention_54_gb300 import inputs
from gpu_helpers import LSE_TOL, O_TOL, assert_close, dev

pytestmark = pytest.mark.gpu


def run_decode(q, k, v, S, scale):
    qd, kd, vd = dev(q, k, v)
    B, H, Sk, D = k.shape
    ws = (torch.empty(B, H, S, D, device="cuda"), torch.empty(B, H, S, device="cuda"),
          torch.empty(B, H, S, device="cuda"))
    o, lse = fa.flash_decode(qd, kd, vd, S, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu(), [w.cpu() for w in ws]


def check_decode(q, k, v, S, scale, what):
    o, lse, (op, mp, lp) = run_decode(q, k, v, S, scale)
    ro, rl = oracle.decode(q, k, v, scale)
    assert_close(o, ro, O_TOL, f"O {what}")
    assert_close(lse, rl[..., 0], LSE_TOL, f"LSE {what}")
    # phase-1 partials: m exact to fp32 rounding, l relative, O_s / l_s like an output
    rop, rmp, rlp = oracle.splitkv_partials(q, k, v, S, scale)
    empty = np.isneginf(rmp)
    assert np.array_equal(np.isneginf(mp.numpy()), empty), "empty partitions differ"
    assert np.all(lp.numpy()[empty] == 0) and np.all(op.numpy()[empty] == 0)
    full = ~empty
    assert_close(mp.numpy()[full], rmp[full], LSE_TOL, f"m_s {what}")
    rel = np.abs(lp.numpy()[full] - rlp[full]) / rlp[full]
    assert rel.max() <= 1e-3, f"l_s {what}: rel err {rel.max():.3e}"
    norm = op.numpy()[full] / lp.numpy()[full][:, None]
    assert_close(norm, rop[full] / rlp[full][:, None], O_TOL, f"O_s/l_s {what}")


def test_decode_workload_full_size():
    w = inputs.WORKLOADS["decode"]
    q, k, v = inputs.make_workload(w)
    check_decode(q, k, v, w.num_splits, w.scale, w.name)


@pytest.mark.parametrize("B,H,Sk,D,dtype,S", [
    (2, 3, 100, 128, torch.bfloat16, 32),   # P = 4: partitions 25..31 empty
    (1, 2, 37, 64, torch.float16, 37),      # one key per partition
    (1, 1, 1, 128, torch.bfloat16, 1),      # a single key
    (2, 2, 1000, 64, torch.float16, 1),     # no split at all
    (1, 4, 4099, 128, torch.float16, 7),    # ragged partitions
    (3, 1, 513, 64, torch.bfloat16, 16),
    (2, 2, 99, 128, torch.bfloat16, 33),    # three keys per partition: lane groups of a warp disagree
    (1, 3, 10, 64, torch.float16, 5),       # two keys per partition, four lane groups per warp
])
def test_decode_shapes(B, H, Sk, D, dtype, S):
    q, k, v = inputs.make_dense(B, H, 1, Sk, D, dtype, seed=Sk + S)
    check_decode(q, k, v, S, 1.0 / math.sqrt(D), f"{(B, H, Sk, D, dtype, S)}")


def test_decode_split_count_does_not_change_the_answer():
    q, k, v = inputs.make_dense(2, 2, 1, 2048, 128, torch.bfloat16, seed=31)
    outs = [run_decode(q, k, v, S, 0.088)[0].float() for S in (1, 8, 32, 1024)]
    for o in outs[1:]:
        assert_close(o, outs[0], 2 * O_TOL, "split count")
