"""The tcgen05 building blocks of the forward kernel, one at a time, against
torch fp32 matmuls: TMA + SS MMA with K-major operands (S = Q K^T), TS MMA with
P in TMEM and V MN-major in smem (O = P V), and the bounded barrier wait."""
import ctypes
import time

import pytest
import torch

from exact_attention_54_gb300 import build as fabuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def st():
    fabuild.build()
    lib = ctypes.CDLL(fabuild.SELFTEST_LIB)
    vp, i, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong
    lib.fa_selftest_qk.argtypes = [vp, vp, vp, i, i, vp, u64, vp]
    lib.fa_selftest_pv.argtypes = [vp, vp, vp, i, i, vp, u64, vp]
    lib.fa_selftest_tn.argtypes = [vp, vp, vp, i, i, vp, u64, vp]
    lib.fa_selftest_watchdog.argtypes = [vp, u64, vp]
    lib.fa_selftest_ldmax.argtypes = [vp, vp, vp, vp]
    return lib


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _diagnose_qk(c, a, b):
    ref = a.float() @ b.float().T
    hyps = {"A B^T": ref, "B A^T": ref.T, "A A^T": a.float() @ a.float().T}
    return {k: float((c - v).abs().max()) for k, v in hyps.items()}


def _diagnose_pv(c, p, v):
    pf, vf = p.float(), v.float()
    swapped = pf.view(128, 64, 2).flip(-1).reshape(128, 128)
    hyps = {"P V": pf @ vf, "P^T V": pf.T @ vf, "pairs swapped": swapped @ vf}
    if vf.shape[1] == 128:
        hyps["P V^T"] = pf @ vf.T
    return {k: float((c - x).abs().max()) for k, x in hyps.items()}


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_qk_mma(st, D, dtype):
    g = torch.Generator().manual_seed(D)
    a = torch.randn(128, D, generator=g).to(dtype).cuda()
    b = torch.randn(128, D, generator=g).to(dtype).cuda()
    c = torch.full((128, 128), float("nan"), device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = st.fa_selftest_qk(a.data_ptr(), b.data_ptr(), c.data_ptr(), D, int(dtype == torch.bfloat16),
                           status.data_ptr(), 1_000_000_000, _stream())
    torch.cuda.synchronize()
    assert rc == 0 and int(status) == 0
    err = float((c - a.float() @ b.float().T).abs().max())
    assert err < 1e-3, _diagnose_qk(c, a, b)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_pv_mma(st, D, dtype):
    g = torch.Generator().manual_seed(100 + D)
    p = torch.rand(128, 128, generator=g).to(dtype).cuda()
    v = torch.randn(128, D, generator=g).to(dtype).cuda()
    c = torch.full((128, D), float("nan"), device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = st.fa_selftest_pv(p.data_ptr(), v.data_ptr(), c.data_ptr(), D, int(dtype == torch.bfloat16),
                           status.data_ptr(), 1_000_000_000, _stream())
    torch.cuda.synchronize()
    assert rc == 0 and int(status) == 0
    err = float((c - p.float() @ v.float()).abs().max())
    assert err < 1e-3, _diagnose_pv(c, p, v)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_transposed_a_mma(st, D, dtype):
    """C = X^T Y with X read as an MN-major A operand (the layout the backward
    pass uses for dQ = dS K with dS^T in shared memory)."""
    g = torch.Generator().manual_seed(200 + D)
    x = torch.randn(128, 128, generator=g).to(dtype).cuda()
    y = torch.randn(128, D, generator=g).to(dtype).cuda()
    c = torch.full((128, D), float("nan"), device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = st.fa_selftest_tn(x.data_ptr(), y.data_ptr(), c.data_ptr(), D, int(dtype == torch.bfloat16),
                           status.data_ptr(), 1_000_000_000, _stream())
    torch.cuda.synchronize()
    assert rc == 0 and int(status) == 0
    ref = x.float().T @ y.float()
    err = float((c - ref).abs().max())
    hyps = {"X^T Y": ref, "X Y": x.float() @ y.float()}
    assert err < 1e-3, {k: float((c - v).abs().max()) for k, v in hyps.items()}


def test_reducing_tmem_load_returns_values_and_row_max(st):
    """The forward's softmax takes each row's maximum from the TMEM loads
    (tcgen05.ld.red max): values must come back unchanged and the maximum
    must be exact, including very large and very negative entries."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(128, 32, generator=g) * 30
    x[5, 7] = 1e30
    x[9, :] = -torch.arange(32, dtype=torch.float32) - 1e20
    x[17, :] = float("-inf")
    x[17, 31] = -2.5
    xd = x.cuda()
    y = torch.full_like(xd, float("nan"))
    mx = torch.full((128,), float("nan"), device="cuda")
    assert st.fa_selftest_ldmax(xd.data_ptr(), y.data_ptr(), mx.data_ptr(), _stream()) == 0
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), x)
    assert torch.equal(mx.cpu(), x.max(dim=1).values)


def test_watchdog_gives_up_and_gpu_stays_usable(st):
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert st.fa_selftest_watchdog(status.data_ptr(), 20_000_000, _stream()) == 0  # 20 ms limit
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status) == 1, "the wait on a barrier nobody arrives at must time out"
    assert 0.015 < dt < 5.0, dt
    # the context is intact and TMEM was released: a real MMA still runs
    a = torch.randn(128, 64, dtype=torch.float16, device="cuda")
    c = torch.empty(128, 128, device="cuda")
    status.fill_(-1)
    assert st.fa_selftest_qk(a.data_ptr(), a.data_ptr(), c.data_ptr(), 64, 0, status.data_ptr(),
                             1_000_000_000, _stream()) == 0
    torch.cuda.synchronize()
    assert int(status) == 0
    assert float((c - a.float() @ a.float().T).abs().max()) < 1e-3
