"""Dense forward (fa_fwd) against the fp64 oracle on the same seeded inputs.

Every shape, the full-size LLaMA-7B prefill (1,32,4096,4096,128, causal,
bf16) in the launch configuration the benchmark times included, is compared
element by element over every row of every head. The masking bookkeeping
is checked exactly: results must not change by a single bit when keys that no
query may see are poisoned."""
import pytest
import torch

import exact_attention_54_gb300 as fa
import oracle
from exact_attention_54_gb300 import inputs
from gpu_helpers import LSE_TOL, O_TOL, assert_close, dev

pytestmark = pytest.mark.gpu


def run(q, k, v, causal, scale):
    qd, kd, vd = dev(q, k, v)
    o, lse = fa.flash_attention(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    return o.cpu(), lse.cpu()


def check(q, k, v, causal, scale, rows=None, what=""):
    o, lse = run(q, k, v, causal, scale)
    ro, rl = oracle.attention(q, k, v, causal, scale, rows=rows)
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    assert_close(o, ro, O_TOL, f"O {what}")
    assert_close(lse, rl, LSE_TOL, f"LSE {what}")


@pytest.mark.parametrize("key", ["tiny", "tiny_causal", "small"])
def test_named_workloads(key):
    w = inputs.WORKLOADS[key]
    q, k, v = inputs.make_workload(w)
    check(q, k, v, w.causal, w.scale, what=w.name)


SHAPES = [
    # B, H, Sq, Sk, D, dtype, causal
    (1, 1, 1, 1, 64, torch.float16, False),
    (1, 1, 1, 1, 128, torch.bfloat16, True),
    (2, 3, 129, 129, 64, torch.bfloat16, True),
    (1, 2, 200, 200, 128, torch.float16, True),
    (1, 2, 300, 77, 128, torch.bfloat16, False),
    (1, 2, 77, 300, 64, torch.float16, False),
    (1, 2, 300, 77, 64, torch.bfloat16, True),     # Sq > Sk: late rows see every key
    (1, 2, 77, 300, 128, torch.float16, True),     # Sq < Sk: top-left alignment
    (2, 2, 640, 640, 128, torch.bfloat16, True),   # several tile pairs, odd tile count
    (1, 1, 1000, 1000, 64, torch.float16, False),
    (3, 2, 384, 512, 128, torch.bfloat16, False),
    # D = 256 (one query tile per CTA, 64-key K/V tiles)
    (1, 1, 1, 1, 256, torch.float16, True),
    (1, 2, 300, 300, 256, torch.bfloat16, True),
    (1, 2, 200, 77, 256, torch.float16, False),
    (2, 1, 129, 500, 256, torch.bfloat16, False),
    (1, 2, 77, 300, 256, torch.float16, True),
    (2, 2, 640, 640, 256, torch.bfloat16, True),
    # D = 512, 1024 (Split-D: 256-column output slices, Q and K streamed)
    (1, 1, 1, 1, 512, torch.float16, True),
    (1, 2, 300, 300, 512, torch.bfloat16, True),
    (2, 1, 129, 500, 512, torch.float16, False),
    (1, 1, 1, 1, 1024, torch.bfloat16, False),
    (1, 2, 200, 77, 1024, torch.float16, False),
    (1, 1, 77, 300, 1024, torch.bfloat16, True),
    (1, 2, 640, 640, 1024, torch.bfloat16, True),
]


@pytest.mark.parametrize("B,H,Sq,Sk,D,dtype,causal", SHAPES)
def test_shapes(B, H, Sq, Sk, D, dtype, causal):
    q, k, v = inputs.make_dense(B, H, Sq, Sk, D, dtype, seed=Sq * 7 + Sk + D)
    check(q, k, v, causal, 1.0 / D ** 0.5, what=f"{(B, H, Sq, Sk, D, dtype, causal)}")


def test_non_default_scale():
    q, k, v = inputs.make_dense(1, 2, 256, 256, 128, torch.bfloat16, seed=5)
    check(q, k, v, True, 0.37, what="scale 0.37")
    check(q, k, v, False, 0.02, what="scale 0.02")


def test_llama_prefill_full_size_all_rows():
    """The LLaMA-7B prefill workload (1,32,4096,4096,128, bf16, causal) in the
    launch configuration the benchmark times: every row of every head against
    the oracle (the oracle runs one head per host thread)."""
    w = inputs.WORKLOADS["llama_prefill"]
    q, k, v = inputs.make_workload(w)
    check(q, k, v, True, w.scale, what=w.name)


def test_d256_workload_full_size_all_rows():
    w = inputs.WORKLOADS["d256"]
    q, k, v = inputs.make_workload(w)
    check(q, k, v, w.causal, w.scale, what=w.name)
    check(q, k, v, True, w.scale, what=w.name + " causal")


@pytest.mark.parametrize("key", ["large_head", "massive_head"])
def test_split_d_workloads_full_size(key):
    """The pages' Split-D rows at full size, every row against the oracle,
    non-causal as printed and causal."""
    w = inputs.WORKLOADS[key]
    q, k, v = inputs.make_workload(w)
    check(q, k, v, w.causal, w.scale, what=w.name)
    check(q, k, v, True, w.scale, what=w.name + " causal")


@pytest.mark.parametrize("D", [512, 1024])
def test_split_d_slices_share_row_statistics(D):
    """Every 256-column slice of a Split-D tile recomputes S = Q K^T over the
    whole head dimension: with V's slices all equal, the slices of O must be
    equal bit for bit (same P, same max, same sum in every CTA)."""
    q, k, v = inputs.make_dense(1, 2, 300, 400, D, torch.bfloat16, seed=17)
    v = v[..., :256].repeat(1, 1, 1, D // 256).contiguous()
    for causal in (False, True):
        o, lse = run(q, k, v, causal, 1.0 / D ** 0.5)
        for s in range(1, D // 256):
            assert torch.equal(o[..., :256].view(torch.int16), o[..., 256 * s:256 * s + 256].view(torch.int16))
        ro, rl = oracle.attention(q, k, v, causal, 1.0 / D ** 0.5)
        assert_close(o, ro, O_TOL, f"O D={D} causal={causal}")
        assert_close(lse, rl, LSE_TOL, f"LSE D={D} causal={causal}")


@pytest.mark.parametrize("D", [128, 256, 512])
def test_causal_skipped_tiles_never_read(D):
    """Causal, Sq = 256 < Sk = 512: keys 256.. are above every row's diagonal,
    so their tiles are skipped. NaN there must not change a single bit."""
    q, k, v = inputs.make_dense(2, 2, 256, 512, D, torch.bfloat16, seed=11)
    o1, l1 = run(q, k, v, True, 0.1)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 256:] = float("nan")
    v2[:, :, 256:] = float("nan")
    o2, l2 = run(q, k2, v2, True, 0.1)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


@pytest.mark.parametrize("D", [64, 256, 1024])
def test_causal_mask_inside_diagonal_tiles_is_exact(D):
    """Rows [0, r) of a causal run depend on keys [0, r) only. With huge K/V
    values planted in keys [r, S) (masked inside the straddling tile), rows
    [0, r) must equal, bit for bit, a run on the first r rows and keys."""
    S, r = 384, 200
    q, k, v = inputs.make_dense(1, 2, S, S, D, torch.float16, seed=12)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, r:] = 3.0e4
    v2[:, :, r:] = -3.0e4
    o_full, l_full = run(q, k2, v2, True, 0.125)
    o_cut, l_cut = run(q[:, :, :r].contiguous(), k[:, :, :r].contiguous(), v[:, :, :r].contiguous(), True, 0.125)
    assert torch.equal(o_full[:, :, :r].view(torch.int16), o_cut.view(torch.int16))
    assert torch.equal(l_full[:, :, :r].view(torch.int32), l_cut.view(torch.int32))


def test_ragged_key_tail_is_masked():
    """Non-causal, Sk = 200: the second key tile is zero-filled past key 199 by
    TMA and must be masked, so the result equals the oracle over 200 keys."""
    q, k, v = inputs.make_dense(1, 1, 128, 200, 64, torch.bfloat16, seed=13)
    check(q, k, v, False, 0.125, what="ragged key tail")


@pytest.mark.parametrize("D", [128, 256, 512])
def test_outputs_do_not_spill_past_the_buffer(D):
    B, H, Sq = 1, 2, 200
    q, k, v = dev(*inputs.make_dense(B, H, Sq, Sq, D, torch.bfloat16, seed=14))
    o_buf = torch.full((B * H * Sq * D + 4096,), 1.5, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * Sq + 256,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[: B * H * Sq * D].view(B, H, Sq, D)
    lse = l_buf[: B * H * Sq].view(B, H, Sq)
    fa.fa_fwd(q, k, v, o, lse, True, 0.1)
    torch.cuda.synchronize()
    assert torch.all(o_buf[B * H * Sq * D:] == 1.5)
    assert torch.all(l_buf[B * H * Sq:] == 7.0)


@pytest.mark.parametrize("D", [64, 128])
def test_output_aligned_to_16_bytes_only(D):
    """O may start 16 bytes past a 32-byte boundary (the entry point asks for
    16-byte alignment); its rows are then written with 16-byte stores instead
    of 32-byte ones. The values must be bit-identical to those written into
    an aligned buffer, nothing outside the view may change, and O must match
    the oracle."""
    B, H, Sq = 1, 2, 200
    q, k, v = inputs.make_dense(B, H, Sq, Sq, D, torch.bfloat16, seed=17)
    qd, kd, vd = dev(q, k, v)
    n = B * H * Sq * D
    o_buf = torch.full((n + 64,), 1.5, dtype=torch.bfloat16, device="cuda")
    o = o_buf[8: 8 + n].view(B, H, Sq, D)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device="cuda")
    fa.fa_fwd(qd, kd, vd, o, lse, True, 0.1)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    assert torch.all(o_buf[:8] == 1.5) and torch.all(o_buf[8 + n:] == 1.5)
    o_al, l_al = fa.flash_attention(qd, kd, vd, causal=True, scale=0.1)
    torch.cuda.synchronize()
    assert o_al.data_ptr() % 32 == 0
    assert torch.equal(o.view(torch.int16), o_al.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), l_al.view(torch.int32))
    ro, rl = oracle.attention(q, k, v, True, 0.1)
    assert_close(o.cpu(), ro, O_TOL, "O at a 16-byte offset")
    assert_close(lse.cpu(), rl, LSE_TOL, "LSE")


def test_repeatable_bitwise():
    q, k, v = inputs.make_dense(2, 4, 512, 512, 128, torch.bfloat16, seed=15)
    o1, l1 = run(q, k, v, True, 0.09)
    o2, l2 = run(q, k, v, True, 0.09)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_non_default_stream():
    q, k, v = dev(*inputs.make_dense(1, 2, 256, 256, 64, torch.float16, seed=16))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.flash_attention(q, k, v, causal=True, scale=0.125, stream=s)
    s.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), True, 0.125)
    assert_close(o.cpu(), ro, O_TOL, "stream O")
    assert_close(lse.cpu(), rl, LSE_TOL, "stream LSE")
