"""The abort path of the prefill kernels, run on the GPU without a fault.

fa_test_withhold_load makes CTA 0 of a launch withhold one tile load, so a
bounded on-chip wait is left that nothing completes (a barrier nobody
arrives at): the wait runs out after a short limit, the CTA drains the copies
it did issue, releases its tensor memory and stops, and the error word reads
FA_ERR_DEVICE_TIMEOUT. Each test then turns the setting off and checks that
the next call on the same context is correct against the oracle (which it
could not be if tensor memory had been left allocated or a copy were still
landing), and that the failed launch wrote nothing outside its outputs."""
import time

import pytest
import torch

import exact_attention_54_gb300 as fa
import oracle
from exact_attention_54_gb300 import inputs
from gpu_helpers import LSE_TOL, O_TOL, assert_close, assert_grad_close, dev

pytestmark = pytest.mark.gpu

FA_ERR_DEVICE_TIMEOUT = -9
LIMIT_NS = 20_000_000  # 20 ms per wait


@pytest.fixture
def withhold():
    yield lambda n: fa.fa_test_withhold_load(n, LIMIT_NS)
    fa.fa_test_withhold_load(0, 0)


def expect_timeout(launch):
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    launch()
    with pytest.raises(fa.FAError) as e:
        fa.fa_check_device_error()
    assert e.value.status == FA_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    fa.fa_test_withhold_load(0, 0)


@pytest.mark.parametrize("D,causal", [(64, False), (128, True), (256, False), (512, False)])
def test_forward_gives_up_and_the_next_call_is_correct(withhold, D, causal):
    B, H, S = 1, 2, 384
    q, k, v = inputs.make_dense(B, H, S, S, D, torch.float16, seed=40 + D)
    qd, kd, vd = dev(q, k, v)
    n = B * H * S * D
    o_buf = torch.full((n + 4096,), 1.5, dtype=torch.float16, device="cuda")
    l_buf = torch.full((B * H * S + 256,), 7.0, dtype=torch.float32, device="cuda")
    o, lse = o_buf[:n].view(B, H, S, D), l_buf[:B * H * S].view(B, H, S)
    withhold(2)  # CTA 0's second V tile
    expect_timeout(lambda: fa.fa_fwd(qd, kd, vd, o, lse, causal, 0.1))
    assert torch.all(o_buf[n:] == 1.5) and torch.all(l_buf[B * H * S:] == 7.0)
    fa.fa_fwd(qd, kd, vd, o, lse, causal, 0.1)
    fa.fa_check_device_error()
    ro, rl = oracle.attention(q, k, v, causal, 0.1)
    assert_close(o.cpu(), ro, O_TOL, "O after an aborted launch")
    assert_close(lse.cpu(), rl, LSE_TOL, "LSE after an aborted launch")


def test_varlen_forward_gives_up_and_the_next_call_is_correct(withhold):
    lengths = [300, 1, 513, 128]
    _, cu, q, k, v = inputs.make_varlen(len(lengths), 0, 0, 2, 128, torch.bfloat16, seed=44, lengths=lengths)
    qd, kd, vd, cud = dev(q, k, v, cu)
    withhold(2)
    expect_timeout(lambda: fa.flash_attention_varlen(qd, kd, vd, cud, cud, max(lengths), causal=True,
                                                     scale=0.09))
    o, lse = fa.flash_attention_varlen(qd, kd, vd, cud, cud, max(lengths), causal=True, scale=0.09)
    fa.fa_check_device_error()
    ro, rl = oracle.attention_varlen(q, k, v, cu, cu, True, 0.09)
    assert_close(o.cpu(), ro, O_TOL, "varlen O after an aborted launch")
    assert_close(lse.cpu(), rl, LSE_TOL, "varlen LSE after an aborted launch")


@pytest.mark.parametrize("D", [64, 128])
def test_backward_gives_up_and_the_next_call_is_correct(withhold, D):
    B, H, S = 1, 2, 384
    q, k, v = inputs.make_dense(B, H, S, S, D, torch.bfloat16, seed=50 + D)
    do = inputs.make_dense(B, H, S, S, D, torch.bfloat16, seed=51 + D)[0]
    qd, kd, vd, dod = dev(q, k, v, do)
    scale = 1.0 / D ** 0.5
    o, lse = fa.flash_attention(qd, kd, vd, causal=True, scale=scale)
    fa.fa_check_device_error()
    withhold(2)  # CTA 0's second Q/dO step
    expect_timeout(lambda: fa.flash_attention_bwd(qd, kd, vd, o, lse, dod, causal=True, scale=scale))
    dq, dk, dv = fa.flash_attention_bwd(qd, kd, vd, o, lse, dod, causal=True, scale=scale)
    fa.fa_check_device_error()
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, True, scale)
    assert_grad_close(dq.cpu(), rq, "dq after an aborted launch")
    assert_grad_close(dk.cpu(), rk, "dk after an aborted launch")
    assert_grad_close(dv.cpu(), rv, "dv after an aborted launch")
