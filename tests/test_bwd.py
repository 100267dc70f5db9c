"""Backward pass (fa_bwd) against the fp64 oracle's gradients on the same
seeded inputs, with the forward's O and LSE from fa_fwd.

Tolerance: the kernel rounds P and dS to 16 bits before their products and
accumulates in fp32, so an element of dQ, dK or dV carries a relative error
of a few 2^-9 of the magnitudes that meet in its sum; the check is
max |g - ref| <= 2e-2 * max(1, max |ref|) per tensor, plus
||g - ref|| <= 1e-2 * max(||ref||, sqrt(n)). Bookkeeping is exact: keys no query can see get
dK = dV = 0 bit for bit, and dK, dV are bitwise repeatable."""
import pytest
import torch

import exact_attention_54_gb300 as fa
import oracle
from exact_attention_54_gb300 import inputs
from gpu_helpers import assert_grad_close, dev

pytestmark = pytest.mark.gpu


def grads(q, k, v, do, causal, scale):
    qd, kd, vd, dod = dev(q, k, v, do)
    o, lse = fa.flash_attention(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.flash_attention_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    return dq.cpu(), dk.cpu(), dv.cpu()


def check(B, H, Sq, Sk, D, dtype, causal, seed, scale=None):
    q, k, v = inputs.make_dense(B, H, Sq, Sk, D, dtype, seed=seed)
    do = inputs.make_dense(B, H, Sq, Sq, D, dtype, seed=seed + 1)[0]
    scale = 1.0 / D ** 0.5 if scale is None else scale
    dq, dk, dv = grads(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal, scale)
    what = f"{(B, H, Sq, Sk, D, dtype, causal)}"
    assert_grad_close(dq, rq, "dq " + what)
    assert_grad_close(dk, rk, "dk " + what)
    assert_grad_close(dv, rv, "dv " + what)
    return dq, dk, dv


SHAPES = [
    # B, H, Sq, Sk, D, dtype, causal
    (1, 1, 1, 1, 64, torch.float16, False),
    (1, 1, 128, 128, 64, torch.float16, False),
    (1, 2, 200, 200, 128, torch.bfloat16, True),
    (2, 2, 300, 77, 64, torch.bfloat16, False),
    (1, 2, 77, 300, 128, torch.float16, False),
    (1, 2, 300, 77, 128, torch.bfloat16, True),    # Sq > Sk: late rows see every key
    (1, 2, 77, 300, 64, torch.float16, True),      # Sq < Sk: keys past the last query get no gradient
    (2, 2, 640, 640, 128, torch.bfloat16, True),
    (1, 3, 384, 512, 64, torch.float16, False),
]


@pytest.mark.parametrize("B,H,Sq,Sk,D,dtype,causal", SHAPES)
def test_bwd_matches_oracle(B, H, Sq, Sk, D, dtype, causal):
    check(B, H, Sq, Sk, D, dtype, causal, seed=Sq * 3 + Sk + D)


def test_bwd_non_default_scale():
    check(1, 2, 256, 256, 128, torch.bfloat16, True, seed=9, scale=0.3)


def test_unreachable_keys_get_exact_zero_and_dk_dv_repeat_bitwise():
    """Causal, Sq = 200 < Sk = 520: keys 200.. are above every query's
    diagonal (and keys 256.. form whole tiles no query visits)."""
    q, k, v = inputs.make_dense(1, 2, 200, 520, 64, torch.bfloat16, seed=61)
    do = inputs.make_dense(1, 2, 200, 200, 64, torch.bfloat16, seed=62)[0]
    dq1, dk1, dv1 = grads(q, k, v, do, True, 0.125)
    assert torch.count_nonzero(dk1[:, :, 200:]) == 0 and torch.count_nonzero(dv1[:, :, 200:]) == 0
    _, dk2, dv2 = grads(q, k, v, do, True, 0.125)
    assert torch.equal(dk1.view(torch.int16), dk2.view(torch.int16))
    assert torch.equal(dv1.view(torch.int16), dv2.view(torch.int16))
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, 0.125)
    assert_grad_close(dq1, rq, "dq")
    assert_grad_close(dk1[:, :, :200], rk[:, :, :200], "dk")


@pytest.mark.parametrize("D", [64, 128])
def test_dk_dv_aligned_to_16_bytes_only(D):
    """dK and dV may start 16 bytes past a 32-byte boundary (the entry point
    asks for 16-byte alignment); their rows are then written with 16-byte
    stores. The values must equal, bit for bit, those written into aligned
    buffers, and nothing outside the views may change."""
    B, H, S = 1, 2, 300
    q, k, v = inputs.make_dense(B, H, S, S, D, torch.bfloat16, seed=63 + D)
    do = inputs.make_dense(B, H, S, S, D, torch.bfloat16, seed=64 + D)[0]
    qd, kd, vd, dod = dev(q, k, v, do)
    o, lse = fa.flash_attention(qd, kd, vd, causal=True, scale=0.1)
    dq_al, dk_al, dv_al = fa.flash_attention_bwd(qd, kd, vd, o, lse, dod, causal=True, scale=0.1)
    n = B * H * S * D
    bufs = [torch.full((n + 64,), 1.5, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dk, dv = (b[8: 8 + n].view(B, H, S, D) for b in bufs)
    assert dk.data_ptr() % 32 == 16 and dv.data_ptr() % 32 == 16
    dq = torch.empty_like(qd)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, S, D) // 4, dtype=torch.float32, device="cuda")
    fa.fa_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, True, 0.1)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    for b in bufs:
        assert torch.all(b[:8] == 1.5) and torch.all(b[8 + n:] == 1.5)
    assert torch.equal(dk.view(torch.int16), dk_al.view(torch.int16))
    assert torch.equal(dv.view(torch.int16), dv_al.view(torch.int16))
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, 0.1)
    assert_grad_close(dk.cpu(), rk, "dk at a 16-byte offset")
    assert_grad_close(dv.cpu(), rv, "dv at a 16-byte offset")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_every_dq_row_written_from_a_nan_workspace(D, causal):
    """dQ and the workspace start out as NaN: the call must clear what it
    accumulates in the workspace and write every dQ row, with a ragged last
    query tile and Sq != Sk."""
    B, H, Sq, Sk = 2, 3, 333, 270
    q, k, v = inputs.make_dense(B, H, Sq, Sk, D, torch.bfloat16, seed=71 + D)
    do = inputs.make_dense(B, H, Sq, Sq, D, torch.bfloat16, seed=72 + D)[0]
    qd, kd, vd, dod = dev(q, k, v, do)
    o, lse = fa.flash_attention(qd, kd, vd, causal=causal, scale=0.1)
    dq = torch.full_like(qd, float("nan"))
    dk, dv = torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.full((fa.fa_bwd_workspace_bytes(B, H, Sq, D) // 4,), float("nan"), dtype=torch.float32,
                    device="cuda")
    fa.fa_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, causal, 0.1)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    assert not torch.isnan(dq).any()
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal, 0.1)
    assert_grad_close(dq.cpu(), rq, f"dq D={D} causal={causal}")
    assert_grad_close(dk.cpu(), rk, f"dk D={D} causal={causal}")


@pytest.mark.parametrize("causal,Sq,Sk", [(True, 300, 700), (False, 333, 260)])
def test_many_units_per_cta_equal_single_head_calls(causal, Sq, Sk):
    """B*H = 160 heads of 3-6 key tiles: the persistent CTAs (one per SM) each
    take several (key tile, head) units in turn, and causal with Sq < Sk
    interleaves units whose keys no query sees. dK and dV of sampled heads
    equal, bit for bit, those of a call on that head alone; dQ, dK and dV
    match the oracle."""
    B, H, D = 4, 40, 128
    q, k, v = inputs.make_dense(B, H, Sq, Sk, D, torch.bfloat16, seed=91)
    do = inputs.make_dense(B, H, Sq, Sq, D, torch.bfloat16, seed=92)[0]
    dq, dk, dv = grads(q, k, v, do, causal, 0.1)
    for b, h in [(0, 0), (1, 17), (3, 39)]:
        one = [x[b:b + 1, h:h + 1].contiguous() for x in (q, k, v, do)]
        _, dk1, dv1 = grads(*one, causal, 0.1)
        assert torch.equal(dk[b:b + 1, h:h + 1].view(torch.int16), dk1.view(torch.int16)), (b, h)
        assert torch.equal(dv[b:b + 1, h:h + 1].view(torch.int16), dv1.view(torch.int16)), (b, h)
        rq, rk, rv = oracle.attention_bwd(*one, causal, 0.1)
        what = f"head ({b}, {h}) causal={causal}"
        assert_grad_close(dq[b:b + 1, h:h + 1], rq, "dq " + what)
        assert_grad_close(dk[b:b + 1, h:h + 1], rk, "dk " + what)
        assert_grad_close(dv[b:b + 1, h:h + 1], rv, "dv " + what)


def test_bwd_llama_prefill_full_size_two_heads():
    """The LLaMA-7B prefill shape (1,32,4096,4096,128, causal, bf16) through
    the full kernel; two heads compared against the oracle (about a minute of
    fp64 CPU work per head)."""
    w = inputs.WORKLOADS["llama_prefill"]
    q, k, v = inputs.make_workload(w)
    do = inputs.make_dense(w.B, w.H, w.Sq, w.Sq, w.D, w.dtype, seed=w.seed + 100)[0]
    dq, dk, dv = grads(q, k, v, do, True, w.scale)
    heads = [0, 17]
    rq, rk, rv = oracle.attention_bwd(q[:, heads], k[:, heads], v[:, heads], do[:, heads], True, w.scale)
    assert_grad_close(dq[:, heads], rq, "dq llama")
    assert_grad_close(dk[:, heads], rk, "dk llama")
    assert_grad_close(dv[:, heads], rv, "dv llama")
