"""The device's f32 -> FP8 E4M3 and f32 -> FP4 E2M1 conversions, which the
cast kernels apply to x * (1 / scale), over every fp32 bit pattern that can
round to a finite code without saturating, against independent encoders:

* E4M3: every non-negative pattern below 464 (the first value that saturates
  whatever the rounding) against PyTorch's CPU float8_e4m3fn cast (the oracle
  encoder is pinned to that cast over the same range); saturation, NaN and
  the sign bit on samples of the rest.
* E2M1: every non-negative pattern below 16 against the oracle's encoder;
  saturation and the sign bit on samples of the rest.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CHUNK = 1 << 26


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_routing_precision_gb300 import _build
    _build.build()
    oracle.build()
    torch.cuda.set_device(0)
    assert ops.device_status() == 0
    yield
    assert ops.device_status() == 0


def _patterns(lo, hi):
    """fp32 values with bit patterns [lo, hi), on the host and the device."""
    bits = torch.arange(lo, hi, dtype=torch.int64).to(torch.int32)
    host = bits.view(torch.float32)
    return host, host.to(DEV)


def _gpu_codes(values_dev, fmt):
    n = values_dev.numel()
    pad = (-n) % 4
    if pad:
        values_dev = torch.cat([values_dev, values_dev.new_zeros(pad)])
    return ops.debug_cvt(values_dev, fmt)[:n].cpu().numpy()


def test_e4m3_every_pattern_below_464_matches_torch():
    end = int(np.float32(464.0).view(np.int32))
    for lo in range(0, end, CHUNK):
        host, dev = _patterns(lo, min(lo + CHUNK, end))
        got = _gpu_codes(dev, ops.CVT_E4M3)
        ref = host.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (f"pattern {lo + bad[0]:#x}: gpu {got[bad[0]]:#04x} "
                               f"torch {ref[bad[0]]:#04x}")


def test_e4m3_saturation_nan_and_sign():
    rng = np.random.default_rng(0)
    big = rng.integers(int(np.float32(464.0).view(np.int32)), 0x7F800000, 1 << 20)
    host = torch.from_numpy(np.concatenate([big, [0x7F800000]]).astype(np.int32)).view(torch.float32)
    assert (_gpu_codes(host.to(DEV), ops.CVT_E4M3) == 0x7E).all()          # +448, +inf too
    nan = torch.from_numpy(rng.integers(0x7F800001, 0x80000000, 4096).astype(np.int32))
    assert (_gpu_codes(nan.view(torch.float32).to(DEV), ops.CVT_E4M3) & 0x7F == 0x7F).all()
    pos = torch.from_numpy(rng.integers(0, 0x7F800000, 1 << 22).astype(np.int32)).view(torch.float32)
    a = _gpu_codes(pos.to(DEV), ops.CVT_E4M3)
    b = _gpu_codes((-pos).to(DEV), ops.CVT_E4M3)
    assert np.array_equal(b, a | 0x80)
    assert _gpu_codes(torch.tensor([-0.0, 0.0, 0.0, 0.0], device=DEV), ops.CVT_E4M3)[0] == 0x80


def test_e2m1_every_pattern_below_16_matches_the_oracle():
    end = int(np.float32(16.0).view(np.int32))
    for lo in range(0, end, CHUNK):
        host, dev = _patterns(lo, min(lo + CHUNK, end))
        got = _gpu_codes(dev, ops.CVT_E2M1)
        ref = oracle.e2m1_encode(host.numpy())
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (f"pattern {lo + bad[0]:#x}: gpu {got[bad[0]]:#x} "
                               f"oracle {ref[bad[0]]:#x}")


def test_e2m1_saturation_and_sign():
    rng = np.random.default_rng(1)
    big = rng.integers(int(np.float32(16.0).view(np.int32)), 0x7F800001, 1 << 20)
    host = torch.from_numpy(big.astype(np.int32)).view(torch.float32)
    assert (_gpu_codes(host.to(DEV), ops.CVT_E2M1) == 7).all()              # +6, +inf too
    pos = torch.from_numpy(rng.integers(0, 0x7F800000, 1 << 22).astype(np.int32)).view(torch.float32)
    a = _gpu_codes(pos.to(DEV), ops.CVT_E2M1)
    b = _gpu_codes((-pos).to(DEV), ops.CVT_E2M1)
    assert np.array_equal(b, a | 8)
    assert _gpu_codes(torch.tensor([-0.0, 0.0, 0.0, 0.0], device=DEV), ops.CVT_E2M1)[0] == 8
