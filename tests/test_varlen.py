"""Packed variable-length forward (fa_fwd_varlen) against the fp64 oracle, plus
exact checks of the sequence bookkeeping: every sequence must equal, bit for
bit, a dense call on its own slice, and nothing may be written outside the
output buffers."""
import pytest
import torch

import exact_attention_54_gb300 as fa
import oracle
from exact_attention_54_gb300 import inputs
from gpu_helpers import LSE_TOL, O_TOL, assert_close, dev

pytestmark = pytest.mark.gpu


def run_varlen(q, k, v, cu, causal, scale):
    qd, kd, vd, cud = dev(q, k, v, cu)
    mx = int((cu[1:] - cu[:-1]).max())
    o, lse = fa.flash_attention_varlen(qd, kd, vd, cud, cud, max(mx, 1), causal=causal, scale=scale)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, torch.float16), (128, torch.bfloat16), (256, torch.float16),
                                     (512, torch.bfloat16)])
def test_small_varlen_all_rows(causal, D, dtype):
    lengths = [1, 127, 128, 129, 0, 300, 5]
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, 3, D, dtype, seed=21, lengths=lengths)
    scale = 1.0 / D ** 0.5
    o, lse = run_varlen(q, k, v, cu, causal, scale)
    ro, rl = oracle.attention_varlen(q, k, v, cu, cu, causal, scale)
    assert_close(o, ro, O_TOL, "varlen O")
    assert_close(lse, rl, LSE_TOL, "varlen LSE")


@pytest.mark.parametrize("D", [128, 256, 1024])
def test_varlen_equals_dense_per_sequence_bitwise(D):
    lengths = [200, 1, 384, 129, 77]
    H = 4
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, H, D, torch.bfloat16, seed=22, lengths=lengths)
    o, lse = run_varlen(q, k, v, cu, True, 0.088)
    for i, L in enumerate(lengths):
        a, b = int(cu[i]), int(cu[i + 1])
        qs, ks, vs = (x[a:b].transpose(0, 1).unsqueeze(0).contiguous() for x in (q, k, v))  # [1,H,L,D]
        qd, kd, vd = dev(qs, ks, vs)
        od, ld = fa.flash_attention(qd, kd, vd, causal=True, scale=0.088)
        torch.cuda.synchronize()
        assert torch.equal(o[a:b].view(torch.int16), od[0].transpose(0, 1).cpu().view(torch.int16)), f"seq {i} O"
        assert torch.equal(lse[:, a:b].view(torch.int32), ld[0].cpu().view(torch.int32)), f"seq {i} LSE"


def test_varlen_guards_untouched():
    lengths = [130, 61, 257]
    H, D = 2, 64
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, H, D, torch.float16, seed=23, lengths=lengths)
    T = int(cu[-1])
    qd, kd, vd, cud = dev(q, k, v, cu)
    o_buf = torch.full(((T + 64) * H * D,), -2.5, dtype=torch.float16, device="cuda")
    l_buf = torch.full((H * T + 300,), 9.0, dtype=torch.float32, device="cuda")
    o = o_buf[: T * H * D].view(T, H, D)
    lse = l_buf[: H * T].view(H, T)
    fa.fa_fwd_varlen(qd, kd, vd, o, lse, cud, cud, max(lengths), True, 0.125)
    torch.cuda.synchronize()
    assert torch.all(o_buf[T * H * D:] == -2.5)
    assert torch.all(l_buf[H * T:] == 9.0)
    ro, rl = oracle.attention_varlen(q, k, v, cu, cu, True, 0.125)
    assert_close(o.cpu(), ro, O_TOL, "guarded O")
    assert_close(lse.cpu(), rl, LSE_TOL, "guarded LSE")


def test_varlen_poison_past_total_is_never_read():
    """Buffers larger than total_tokens hold NaN past the end; the tensor maps
    stop at total, so no NaN may reach any output."""
    lengths = [100, 200]
    H, D = 2, 128
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, H, D, torch.bfloat16, seed=24, lengths=lengths)
    T = int(cu[-1])
    pad = torch.full((128, H, D), float("nan"), dtype=torch.bfloat16)
    kp, vp = torch.cat([k, pad]), torch.cat([v, pad])
    qd, kd, vd, cud = dev(q, kp, vp, cu)
    o, lse = fa.flash_attention_varlen(qd, kd[:T], vd[:T], cud, cud, 200, causal=False, scale=0.1)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_varlen(q, k, v, cu, cu, False, 0.1)
    assert_close(o.cpu(), ro, O_TOL, "poisoned tail O")
    assert_close(lse.cpu(), rl, LSE_TOL, "poisoned tail LSE")


def test_varlen_workload_all_rows():
    """16 sequences, lengths uniform on [64, 2048], H=16, D=128, bf16, causal:
    every row of every sequence and head against the oracle."""
    w = inputs.WORKLOADS["varlen"]
    lengths, cu, q, k, v = inputs.make_workload(w)
    o, lse = run_varlen(q, k, v, cu, w.causal, w.scale)
    ro, rl = oracle.attention_varlen(q, k, v, cu, cu, w.causal, w.scale)
    assert_close(o, ro, O_TOL, "varlen workload O")
    assert_close(lse, rl, LSE_TOL, "varlen workload LSE")


@pytest.mark.parametrize("D", [128, 256])
def test_inconsistent_offsets_compute_nothing_and_report(D):
    """cu_seqlens are only readable on the device. A query sequence longer
    than max_seqlen_q, or offsets past the tensors' token counts, must leave
    O and LSE untouched (no out-of-range reads or writes) and make
    fa_check_device_error report FA_ERR_DEVICE_SEQLENS; the next valid call
    works."""
    H = 2
    lengths = [100, 300]
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, H, D, torch.bfloat16, seed=25, lengths=lengths)
    qd, kd, vd, cud = dev(q, k, v, cu.to(torch.int32))
    T = int(cu[-1])
    cases = {
        "longer than max_seqlen_q": (qd, kd, vd, 200),
        "offsets past total_q/total_k": (qd[:250].contiguous(), kd[:250].contiguous(), vd[:250].contiguous(), 300),
    }
    for what, (qq, kk, vv, mx) in cases.items():
        o = torch.full_like(qq, 3.0)
        lse = torch.full((H, qq.shape[0]), 5.0, dtype=torch.float32, device="cuda")
        fa.fa_fwd_varlen(qq, kk, vv, o, lse, cud, cud, mx, True, 0.1)
        with pytest.raises(fa.FAError) as e:
            fa.fa_check_device_error()
        assert e.value.status == -13, what
        assert torch.all(o == 3.0), what
        assert torch.all(lse == 5.0), what
    o, lse = fa.flash_attention_varlen(qd, kd, vd, cud, cud, 300, causal=True, scale=0.1)
    fa.fa_check_device_error()
    ro, rl = oracle.attention_varlen(q, k, v, cu, cu, True, 0.1)
    assert_close(o.cpu(), ro, O_TOL, "O after the rejected launches")
    assert_close(lse.cpu(), rl, LSE_TOL, "LSE after the rejected launches")
    assert T == 400


@pytest.mark.parametrize("num_seqs", [300, 40])
def test_varlen_schedule_table_and_fallback(num_seqs):
    """The kernel schedules packed sequences from a table it builds from
    cu_seqlens (up to 256 sequences) and falls back to enumerating every
    (pair, sequence, head) beyond that: both must give the oracle's result,
    with empty and one-token sequences mixed in."""
    g = torch.Generator().manual_seed(31 + num_seqs)
    lengths = torch.randint(0, 400 if num_seqs < 256 else 60, (num_seqs,), generator=g)
    lengths[::7] = 0
    lengths[3::11] = 1
    _, cu, q, k, v = inputs.make_varlen(num_seqs, 0, 0, 2, 64, torch.bfloat16, seed=33, lengths=lengths.tolist())
    for causal in (True, False):
        o, lse = run_varlen(q, k, v, cu, causal, 0.125)
        ro, rl = oracle.attention_varlen(q, k, v, cu, cu, causal, 0.125)
        assert_close(o, ro, O_TOL, f"varlen O {num_seqs} causal={causal}")
        assert_close(lse, rl, LSE_TOL, f"varlen LSE {num_seqs} causal={causal}")


def test_varlen_more_items_per_cta_than_cached_records():
    """Each CTA keeps at most 48 of its work items as cached records; with
    8000 items (200 short sequences x 40 heads) a CTA has more rounds than
    that on any GPU of up to 166 SMs, and the kernel resolves every item from
    the schedule table instead. Both forms must give the oracle's result."""
    g = torch.Generator().manual_seed(41)
    lengths = torch.randint(1, 257, (200,), generator=g)
    _, cu, q, k, v = inputs.make_varlen(200, 0, 0, 40, 64, torch.bfloat16, seed=42, lengths=lengths.tolist())
    for causal in (True, False):
        o, lse = run_varlen(q, k, v, cu, causal, 0.125)
        ro, rl = oracle.attention_varlen(q, k, v, cu, cu, causal, 0.125)
        assert_close(o, ro, O_TOL, f"many-item varlen O causal={causal}")
        assert_close(lse, rl, LSE_TOL, f"many-item varlen LSE causal={causal}")
