"""Split-KV decoding over a paged KV cache (fa_decode_paged_splitkv +
fa_splitkv_merge, and the one-launch fa_decode_paged_splitkv_fused) against
the oracle's gather-then-attend definition, plus exact checks of the page
bookkeeping."""
import numpy as np
import pytest
import torch

import exact_attention_54_gb300 as fa
import oracle
from exact_attention_54_gb300 import inputs
from gpu_helpers import LSE_TOL, O_TOL, assert_close, dev

pytestmark = pytest.mark.gpu


def run_paged(q, kc, vc, bt, sl, S, scale):
    qd, kd, vd, btd, sld = dev(q, kc, vc, bt, sl)
    B, H = q.shape[:2]
    D = kc.shape[3]
    ws = (torch.empty(B, H, S, D, device="cuda"), torch.empty(B, H, S, device="cuda"),
          torch.empty(B, H, S, device="cuda"))
    o, lse = fa.flash_decode_paged(qd, kd, vd, btd, sld, S, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    return o.cpu(), lse.cpu(), [w.cpu() for w in ws]


@pytest.mark.parametrize("D,dtype,bs,lens,S", [
    (128, torch.bfloat16, 16, [1000, 1, 0, 257], 8),
    (64, torch.float16, 64, [64, 65, 4096], 16),
    (128, torch.float16, 1, [37, 5], 37),
    (64, torch.bfloat16, 256, [300, 1023, 2], 3),
])
def test_paged_matches_oracle(D, dtype, bs, lens, S):
    B, H = len(lens), 3
    q, kc, vc, bt, sl = inputs.make_paged(B, H, D, bs, lens, dtype, seed=sum(lens) + bs)
    scale = 1.0 / D ** 0.5
    o, lse, (op, mp, lp) = run_paged(q, kc, vc, bt, sl, S, scale)
    ro, rl = oracle.decode_paged(q, kc, vc, bt, sl, scale)
    assert_close(o, ro, O_TOL, "paged O")
    assert_close(lse, rl[..., 0], LSE_TOL, "paged LSE")
    ks = oracle.get().paged_gather(kc, bt, sl)
    vs = oracle.get().paged_gather(vc, bt, sl)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(mp[b].numpy() == -np.inf) and np.all(lp[b].numpy() == 0)
            continue
        rop, rmp, rlp = oracle.splitkv_partials(q[b], ks[b], vs[b], S, scale)
        full = ~np.isneginf(rmp)
        assert np.array_equal(~np.isneginf(mp[b].numpy()), full)
        assert_close(mp[b].numpy()[full], rmp[full], LSE_TOL, f"paged m_s seq {b}")
        rel = np.abs(lp[b].numpy()[full] - rlp[full]) / rlp[full]
        assert rel.max() <= 1e-3


def test_paged_with_one_page_per_sequence_equals_dense_bitwise():
    """block_size = Sk and page b for sequence b make the paged cache the dense
    [B,H,Sk,D] tensor itself: partials and outputs must match bit for bit."""
    B, H, Sk, D, S = 4, 2, 512, 128, 8
    q, k, v = inputs.make_dense(B, H, 1, Sk, D, torch.bfloat16, seed=41)
    bt = torch.arange(B, dtype=torch.int32).reshape(B, 1)
    sl = torch.full((B,), Sk, dtype=torch.int32)
    o_p, l_p, (op_p, mp_p, lp_p) = run_paged(q, k, v, bt, sl, S, 0.088)
    qd, kd, vd = dev(q, k, v)
    ws = (torch.empty(B, H, S, D, device="cuda"), torch.empty(B, H, S, device="cuda"),
          torch.empty(B, H, S, device="cuda"))
    o_d, l_d = fa.flash_decode(qd, kd, vd, S, scale=0.088, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(op_p.view(torch.int32), ws[0].cpu().view(torch.int32))
    assert torch.equal(mp_p.view(torch.int32), ws[1].cpu().view(torch.int32))
    assert torch.equal(lp_p.view(torch.int32), ws[2].cpu().view(torch.int32))
    assert torch.equal(o_p.view(torch.int16), o_d.cpu().view(torch.int16))
    assert torch.equal(l_p.view(torch.int32), l_d.cpu().view(torch.int32))


def test_shared_prefix_page():
    """Two sequences whose first logical block is the same physical page."""
    q, kc, vc, bt, sl = inputs.make_paged(2, 2, 128, 16, [40, 40], torch.bfloat16, seed=43)
    bt[1, 0] = bt[0, 0]
    o, lse, _ = run_paged(q, kc, vc, bt, sl, 4, 0.1)
    ro, rl = oracle.decode_paged(q, kc, vc, bt, sl, 0.1)
    assert_close(o, ro, O_TOL, "shared page O")
    assert_close(lse, rl[..., 0], LSE_TOL, "shared page LSE")


def test_out_of_range_page_is_flagged_not_read():
    """A table entry past num_blocks inside a sequence: the kernel skips that
    page (never dereferences it) and the error word reports it."""
    q, kc, vc, bt, sl = inputs.make_paged(2, 2, 64, 16, [64, 64], torch.float16, seed=44)
    bad = bt.clone()
    bad[1, 2] = kc.shape[0] + 5
    qd, kd, vd, btd, sld = dev(q, kc, vc, bad, sl)
    fa.flash_decode_paged(qd, kd, vd, btd, sld, 4, scale=0.125)
    with pytest.raises(fa.FAError) as e:
        fa.fa_check_device_error()
    assert e.value.status == -11
    fa.fa_check_device_error()  # the word was cleared and the context still works
    o, lse, _ = run_paged(q, kc, vc, bt, sl, 4, 0.125)
    ro, rl = oracle.decode_paged(q, kc, vc, bt, sl, 0.125)
    assert_close(o, ro, O_TOL, "after a flagged call")


def test_paged_workload_full_size():
    w = inputs.WORKLOADS["paged_decode"]
    q, kc, vc, bt, sl = inputs.make_workload(w)
    o, lse, _ = run_paged(q, kc, vc, bt, sl, w.num_splits, w.scale)
    ro, rl = oracle.decode_paged(q, kc, vc, bt, sl, w.scale)
    assert_close(o, ro, O_TOL, f"O {w.name}")
    assert_close(lse, rl[..., 0], LSE_TOL, f"LSE {w.name}")


@pytest.mark.parametrize("D,dtype,bs,lens,S", [
    (128, torch.bfloat16, 16, [1000, 1, 0, 257], 8),
    (64, torch.float16, 64, [64, 65, 4096], 16),
])
def test_paged_fused_matches_oracle_and_two_launch_path(D, dtype, bs, lens, S):
    B, H = len(lens), 3
    q, kc, vc, bt, sl = inputs.make_paged(B, H, D, bs, lens, dtype, seed=sum(lens) + bs + 1)
    scale = 1.0 / D ** 0.5
    qd, kd, vd, btd, sld = dev(q, kc, vc, bt, sl)
    cnt = torch.zeros(B * H, dtype=torch.int32, device="cuda")
    ws = (torch.empty(B, H, S, D, device="cuda"), torch.empty(B, H, S, device="cuda"),
          torch.empty(B, H, S, device="cuda"), cnt)
    o, lse = fa.flash_decode_paged(qd, kd, vd, btd, sld, S, scale=scale, workspace=ws, fused=True)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    assert torch.count_nonzero(cnt) == 0
    ro, rl = oracle.decode_paged(q, kc, vc, bt, sl, scale)
    assert_close(o.cpu(), ro, O_TOL, "paged fused O")
    assert_close(lse.cpu(), rl[..., 0], LSE_TOL, "paged fused LSE")
    o2, lse2, (op2, mp2, lp2) = run_paged(q, kc, vc, bt, sl, S, scale)
    assert torch.equal(ws[0].cpu().view(torch.int32), op2.view(torch.int32))
    assert torch.equal(ws[1].cpu().view(torch.int32), mp2.view(torch.int32))
    assert torch.equal(ws[2].cpu().view(torch.int32), lp2.view(torch.int32))


def test_paged_fused_workload_full_size():
    w = inputs.WORKLOADS["paged_decode"]
    q, kc, vc, bt, sl = inputs.make_workload(w)
    qd, kd, vd, btd, sld = dev(q, kc, vc, bt, sl)
    o, lse = fa.flash_decode_paged(qd, kd, vd, btd, sld, w.num_splits, scale=w.scale, fused=True)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    ro, rl = oracle.decode_paged(q, kc, vc, bt, sl, w.scale)
    assert_close(o.cpu(), ro, O_TOL, f"fused O {w.name}")
    assert_close(lse.cpu(), rl[..., 0], LSE_TOL, f"fused LSE {w.name}")
