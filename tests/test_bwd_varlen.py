"""Backward pass over packed sequences (fa_bwd_varlen) against the fp64
oracle's per-sequence gradients, with the forward's O and LSE from
fa_fwd_varlen; the same tolerance as the dense backward (tests/test_bwd.py).
Bookkeeping is exact: keys of a sequence without queries get dK = dV = 0 bit
for bit, and a sequence's dK and dV equal, bit for bit, those of a dense
fa_bwd call on that sequence alone."""
import pytest
import torch

import exact_attention_54_gb300 as fa
import oracle
from exact_attention_54_gb300 import inputs
from gpu_helpers import assert_grad_close, dev

pytestmark = pytest.mark.gpu


def _cu(lengths):
    return inputs.cu_from_lengths(lengths)


def run(q, k, v, do, cu_q, cu_k, causal, scale, max_q=None, max_k=None):
    qd, kd, vd, dod, cqd, ckd = dev(q, k, v, do, cu_q, cu_k)
    lq = (cu_q[1:] - cu_q[:-1])
    lk = (cu_k[1:] - cu_k[:-1])
    mq = max(int(lq.max()), 1) if max_q is None else max_q
    mk = max(int(lk.max()), 1) if max_k is None else max_k
    o, lse = fa.flash_attention_varlen(qd, kd, vd, cqd, ckd, mq, causal=causal, scale=scale)
    dq, dk, dv = fa.flash_attention_varlen_bwd(qd, kd, vd, o, lse, dod, cqd, ckd, mq, mk, causal=causal, scale=scale)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    return dq.cpu(), dk.cpu(), dv.cpu()


def check(q, k, v, do, cu_q, cu_k, causal, scale, what):
    got = run(q, k, v, do, cu_q, cu_k, causal, scale)
    ref = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k, causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert_grad_close(g, r, f"{name} {what}")
    return got


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, torch.float16), (128, torch.bfloat16), (64, torch.bfloat16),
                                     (128, torch.float16)])
def test_small_varlen_bwd_all_rows(causal, D, dtype):
    lengths = [1, 127, 128, 129, 0, 300, 5]
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, 3, D, dtype, seed=61, lengths=lengths)
    do = inputs.make_varlen(len(lengths), 0, 0, 3, D, dtype, seed=62, lengths=lengths)[2]
    check(q, k, v, do, cu, cu, causal, 1.0 / D ** 0.5, f"D={D} {dtype} causal={causal}")


@pytest.mark.parametrize("D", [64, 128])
def test_varlen_bwd_query_and_key_lengths_differ(D):
    """cu_seqlens_q != cu_seqlens_k (top-left causal inside each sequence), with
    a sequence that has keys but no queries: its keys get exact zeros."""
    Lq, Lk = [50, 200, 0, 130, 7], [70, 150, 40, 300, 7]
    H = 2
    cq, ck = _cu(Lq), _cu(Lk)
    g = torch.Generator().manual_seed(63)
    q = inputs.randn((int(cq[-1]), H, D), torch.bfloat16, g)
    do = inputs.randn((int(cq[-1]), H, D), torch.bfloat16, g)
    k = inputs.randn((int(ck[-1]), H, D), torch.bfloat16, g)
    v = inputs.randn((int(ck[-1]), H, D), torch.bfloat16, g)
    for causal in (False, True):
        _, dk, dv = check(q, k, v, do, cq, ck, causal, 0.1, f"D={D} causal={causal}")
        a, b = int(ck[2]), int(ck[3])
        assert torch.all(dk[a:b] == 0) and torch.all(dv[a:b] == 0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_varlen_bwd_queries_without_keys_get_zero_dq(D, causal):
    """A sequence with queries but no keys: dS is empty there, so its dQ rows
    are exactly zero. dQ and the workspace start out as NaN, so every dQ row
    has to be written by the call; the other sequences match the oracle. The
    keyless sequence's O and LSE are set to the empty-set values (0, -inf)."""
    Lq, Lk = [40, 70, 0, 100], [60, 0, 30, 129]
    H = 2
    cq, ck = _cu(Lq), _cu(Lk)
    g = torch.Generator().manual_seed(81)
    q = inputs.randn((int(cq[-1]), H, D), torch.bfloat16, g)
    do = inputs.randn((int(cq[-1]), H, D), torch.bfloat16, g)
    k = inputs.randn((int(ck[-1]), H, D), torch.bfloat16, g)
    v = inputs.randn((int(ck[-1]), H, D), torch.bfloat16, g)
    qd, kd, vd, dod, cqd, ckd = dev(q, k, v, do, cq, ck)
    o, lse = fa.flash_attention_varlen(qd, kd, vd, cqd, ckd, max(Lq), causal=causal, scale=0.1)
    a, b = int(cq[1]), int(cq[2])
    o[a:b] = 0
    lse[:, a:b] = float("-inf")
    dq = torch.full_like(qd, float("nan"))
    dk, dv = torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.full((fa.fa_bwd_varlen_workspace_bytes(qd.shape[0], H, D) // 4,), float("nan"),
                    dtype=torch.float32, device="cuda")
    fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, cqd, ckd, max(Lq), max(Lk), causal, 0.1)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    dq = dq.cpu()
    assert torch.all(dq[a:b] == 0)
    rq, rk, rv = oracle.attention_bwd_varlen(q, k, v, do, cq, ck, causal, 0.1)
    assert_grad_close(dq, rq, f"dq D={D} causal={causal}")
    assert_grad_close(dk.cpu(), rk, f"dk D={D} causal={causal}")
    assert_grad_close(dv.cpu(), rv, f"dv D={D} causal={causal}")


def test_varlen_bwd_dk_dv_equal_dense_per_sequence_bitwise():
    lengths = [200, 1, 384, 129, 77]
    H, D = 2, 128
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, H, D, torch.bfloat16, seed=64, lengths=lengths)
    do = inputs.make_varlen(len(lengths), 0, 0, H, D, torch.bfloat16, seed=65, lengths=lengths)[2]
    dq, dk, dv = run(q, k, v, do, cu, cu, True, 0.088)
    for i in range(len(lengths)):
        a, b = int(cu[i]), int(cu[i + 1])
        qs, ks, vs, dos = (x[a:b].transpose(0, 1).unsqueeze(0).contiguous() for x in (q, k, v, do))  # [1,H,L,D]
        qd, kd, vd, dod = dev(qs, ks, vs, dos)
        o, lse = fa.flash_attention(qd, kd, vd, causal=True, scale=0.088)
        rq, rk, rv = fa.flash_attention_bwd(qd, kd, vd, o, lse, dod, causal=True, scale=0.088)
        torch.cuda.synchronize()
        assert torch.equal(dk[a:b].view(torch.int16), rk[0].transpose(0, 1).cpu().view(torch.int16)), f"seq {i} dK"
        assert torch.equal(dv[a:b].view(torch.int16), rv[0].transpose(0, 1).cpu().view(torch.int16)), f"seq {i} dV"
        assert_grad_close(dq[a:b], rq[0].transpose(0, 1).cpu().double().numpy(), f"seq {i} dQ vs dense")


def test_varlen_bwd_workload_all_rows():
    """The packed-sequence workload (16 sequences of 64-2048 tokens, H=16,
    D=128, bf16, causal): every gradient row against the oracle."""
    w = inputs.WORKLOADS["varlen"]
    lengths, cu, q, k, v = inputs.make_workload(w)
    do = inputs.make_varlen(w.num_seqs, 0, 0, w.H, w.D, w.dtype, seed=w.seed + 100, lengths=lengths.tolist())[2]
    check(q, k, v, do, cu, cu, True, w.scale, w.name)


def test_varlen_bwd_inconsistent_offsets_report():
    """A sequence longer than max_seqlen_k (or _q) is skipped and reported as
    FA_ERR_DEVICE_SEQLENS; the next valid call works."""
    lengths = [100, 300]
    H, D = 2, 64
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, H, D, torch.bfloat16, seed=66, lengths=lengths)
    do = inputs.make_varlen(len(lengths), 0, 0, H, D, torch.bfloat16, seed=67, lengths=lengths)[2]
    qd, kd, vd, dod, cud = dev(q, k, v, do, cu)
    o, lse = fa.flash_attention_varlen(qd, kd, vd, cud, cud, 300, causal=True, scale=0.1)
    fa.fa_check_device_error()
    for mq, mk in ((200, 300), (300, 200)):
        dq, dk, dv = (torch.zeros_like(x) for x in (qd, kd, vd))
        ws = torch.empty(fa.fa_bwd_varlen_workspace_bytes(qd.shape[0], H, D) // 4, dtype=torch.float32,
                         device="cuda")
        fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, cud, cud, mq, mk, True, 0.1)
        with pytest.raises(fa.FAError) as e:
            fa.fa_check_device_error()
        assert e.value.status == -13
    run(q, k, v, do, cu, cu, True, 0.1)
