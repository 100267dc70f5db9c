"""The benchmark's FLOP convention reproduces the TFLOPS the pages print."""
import os

from exact_attention_54_gb300.metrics import attention_flops, decode_bytes, varlen_flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_benchmarks.txt")


def _rows():
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            label, *nums = line.split()
            B, H, Sq, Sk, D = (int(x) for x in nums[:5])
            yield label, B, H, Sq, Sk, D, float(nums[5]), float(nums[6])


def test_page_tflops_reproduced():
    rows = list(_rows())
    assert len(rows) == 6
    for label, B, H, Sq, Sk, D, ms, printed in rows:
        tflops = attention_flops(B, H, Sq, Sk, D, causal=False) / (ms * 1e-3) / 1e12
        assert abs(tflops - printed) <= 0.005 + 1e-9, (label, tflops, printed)


def test_causal_and_varlen_counts():
    assert attention_flops(1, 32, 4096, 4096, 128, True) == 2 * 32 * 4096 * 4096 * 128
    assert varlen_flops([3, 5], [3, 5], 2, 4, False) == 4 * (9 + 25) * 2 * 4
    assert varlen_flops([3, 5], [3, 5], 2, 4, True) == 2 * (9 + 25) * 2 * 4
    # decode: K+V for B*H heads of Sk keys, plus q and O, 2 bytes each
    assert decode_bytes(16, 8, 8192, 128) == 16 * 8 * (2 * 8192 * 128 + 2 * 128) * 2
