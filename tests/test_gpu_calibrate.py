"""kv4_calibrate_global_scale on the GPU against the oracle's calibration:
the scales must be the same FP32 values (the maximum is exact, the division
correctly rounded)."""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
from kv4_testlib import dev_bf16
from oracle import quant as Q
from workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def _run(k, v):
    out = torch.full((2,), -5.0, dtype=torch.float32, device="cuda")
    K.kv4_calibrate_global_scale(dev_bf16(k), dev_bf16(v), out)
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("T,H,D", [(1, 1, 64), (1000, 4, 128), (4097, 2, 256)])
def test_calibrate_matches_oracle(T, H, D):
    rng = np.random.default_rng(T + D)
    k = f32_to_bf16_bits(rng.standard_normal((T, H, D)).astype(np.float32) * 3)
    v = f32_to_bf16_bits(rng.standard_normal((T, H, D)).astype(np.float32) * 0.01)
    v[T // 2, H - 1, D - 3] = f32_to_bf16_bits(np.array([-97.25], np.float32))[0]   # one outlier
    got = _run(k, v)
    assert got[0] == Q.calibrate_global_scale(k) and got[1] == Q.calibrate_global_scale(v)


def test_calibrate_zero_and_empty():
    z = np.zeros((16, 2, 64), np.uint16)
    assert _run(z, z).tolist() == [1.0, 1.0]
    e = np.zeros((0, 2, 64), np.uint16)
    out = torch.zeros(2, dtype=torch.float32, device="cuda")
    K.kv4_calibrate_global_scale(torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda"),
                                 torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda"), out)
    assert out.cpu().tolist() == [1.0, 1.0]
    del e
