"""Split-KV decoding (fa_decode_splitkv + fa_splitkv_merge, and the one-launch
fa_decode_splitkv_fused) against the fp64 oracle: the merged output against
full single-query attention, and the phase-1 partials against the oracle's own
partials (uneven and empty partitions included)."""
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


def run_fused(q, k, v, S, scale, counters=None, stream=None):
    qd, kd, vd = dev(q, k, v)
    B, H, Sk, D = k.shape
    ws = (torch.empty(B, H, S, D, device="cuda"), torch.empty(B, H, S, device="cuda"),
          torch.empty(B, H, S, device="cuda"),
          torch.zeros(B * H, dtype=torch.int32, device="cuda") if counters is None else counters)
    o, lse = fa.flash_decode(qd, kd, vd, S, scale=scale, workspace=ws, fused=True, stream=stream)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu(), [w.cpu() for w in ws]


@pytest.mark.parametrize("B,H,Sk,D,dtype,S", [
    (16, 8, 8192, 128, torch.bfloat16, 32),  # the decode workload's shape
    (2, 3, 100, 128, torch.bfloat16, 32),    # empty partitions
    (1, 2, 37, 64, torch.float16, 37),
    (1, 1, 1, 128, torch.bfloat16, 1),
    (3, 1, 513, 64, torch.bfloat16, 16),
    (1, 2, 5000, 128, torch.float16, 1024),  # the most partitions one call takes
])
def test_fused_matches_oracle_and_two_launch_path(B, H, Sk, D, dtype, S):
    q, k, v = inputs.make_dense(B, H, 1, Sk, D, dtype, seed=7 * Sk + S)
    scale = 1.0 / math.sqrt(D)
    o, lse, (op, mp, lp, cnt) = run_fused(q, k, v, S, scale)
    ro, rl = oracle.decode(q, k, v, scale)
    assert_close(o, ro, O_TOL, "fused O")
    assert_close(lse, rl[..., 0], LSE_TOL, "fused LSE")
    assert torch.count_nonzero(cnt) == 0, "counters must be left at zero"
    # phase 1 is the same code in both paths: partials agree bit for bit
    o2, lse2, (op2, mp2, lp2) = run_decode(q, k, v, S, scale)
    assert torch.equal(op.view(torch.int32), op2.view(torch.int32))
    assert torch.equal(mp.view(torch.int32), mp2.view(torch.int32))
    assert torch.equal(lp.view(torch.int32), lp2.view(torch.int32))
    assert_close(o.float(), o2.float(), O_TOL, "fused vs two-launch O")
    assert_close(lse, lse2, LSE_TOL, "fused vs two-launch LSE")


def test_fused_counters_rearm_across_calls_and_streams():
    """The same counters serve back-to-back calls (on two streams, ordered by
    an event) without being cleared in between."""
    q, k, v = inputs.make_dense(4, 4, 1, 3000, 128, torch.bfloat16, seed=77)
    qd, kd, vd = dev(q, k, v)
    cnt = torch.zeros(16, dtype=torch.int32, device="cuda")
    ws = (torch.empty(4, 4, 24, 128, device="cuda"), torch.empty(4, 4, 24, device="cuda"),
          torch.empty(4, 4, 24, device="cuda"), cnt)
    outs = []
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for st in (s1, s2, s1):
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            o, lse = fa.flash_decode(qd, kd, vd, 24, scale=0.09, workspace=ws, fused=True, stream=st)
        torch.cuda.current_stream().wait_stream(st)
        outs.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert torch.count_nonzero(cnt) == 0
    for o, lse in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(lse.view(torch.int32), outs[0][1].view(torch.int32))
    ro, rl = oracle.decode(q, k, v, 0.09)
    assert_close(outs[0][0].cpu(), ro, O_TOL, "fused O")
