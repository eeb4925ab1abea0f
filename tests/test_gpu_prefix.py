"""kv4_dequant_prefix on the GPU against the oracle: FP8 workspace bytes must
match exactly (NVFP4 and INT4, ragged prefixes, zero-length prefixes)."""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
import oracle
from kv4_testlib import Case, assert_guard_intact, guarded_empty

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
@pytest.mark.parametrize("D", [64, 256])
def test_prefix_bit_exact(fmt, D):
    c = Case(fmt, 2, 4, D, [300, 17, 0, 129], 16 if D == 64 else 64, seed=11 + D)
    prefix = np.array([250, 17, 0, 1], np.int32)
    cu = np.concatenate([[0], np.cumsum(prefix)]).astype(np.int64)
    s8 = (6 * c.g).astype(np.float32) if fmt == "nvfp4" else np.array([0.01, 0.02], np.float32)
    spec, ref_pool = c.oracle_pool()
    wk, wv = oracle.attention.dequant_prefix(ref_pool, spec, c.g, c.table, prefix, s8)
    pool = c.gpu_pool()
    total = int(prefix.sum())
    gk, gk_guard = guarded_empty((total, c.Hkv, D), 0xEE)
    gv, gv_guard = guarded_empty((total, c.Hkv, D), 0xEE)
    K.kv4_dequant_prefix(pool, c.d_g, torch.from_numpy(c.table).cuda(), torch.from_numpy(prefix).cuda(),
                         torch.from_numpy(cu).cuda(), int(prefix.max()), torch.from_numpy(s8).cuda(), gk, gv)
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert np.array_equal(gk.cpu().numpy(), wk)
    assert np.array_equal(gv.cpu().numpy(), wv)
    assert_guard_intact(gk_guard, "K workspace")
    assert_guard_intact(gv_guard, "V workspace")
    assert_guard_intact(pool.guard, "pool")


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
def test_prefix_rows_on_and_off_a_128_byte_boundary(fmt):
    """Head dim 64 and three KV heads: a request's first workspace row starts
    64 bytes into a 128-byte row when its token offset is odd, and then its
    outputs are stored by the lanes instead of by the tensor copy; requests
    at offsets 0 and 32 take the copy (at a non-zero row).  Whole workspaces
    compared, with guard bytes after them."""
    c = Case(fmt, 3, 6, 64, [40, 64, 130], 16, seed=5)
    prefix = np.array([32, 33, 129], np.int32)        # offsets 0, 32, 65
    cu = np.concatenate([[0], np.cumsum(prefix)]).astype(np.int64)
    s8 = (6 * c.g).astype(np.float32) if fmt == "nvfp4" else np.array([0.01, 0.02], np.float32)
    spec, ref_pool = c.oracle_pool()
    wk, wv = oracle.attention.dequant_prefix(ref_pool, spec, c.g, c.table, prefix, s8)
    pool = c.gpu_pool()
    total = int(prefix.sum())
    gk, gk_guard = guarded_empty((total, c.Hkv, 64), 0xEE)
    gv, gv_guard = guarded_empty((total, c.Hkv, 64), 0xEE)
    K.kv4_dequant_prefix(pool, c.d_g, torch.from_numpy(c.table).cuda(), torch.from_numpy(prefix).cuda(),
                         torch.from_numpy(cu).cuda(), int(prefix.max()), torch.from_numpy(s8).cuda(), gk, gv)
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert np.array_equal(gk.cpu().numpy(), wk)
    assert np.array_equal(gv.cpu().numpy(), wv)
    assert_guard_intact(gk_guard, "K workspace")
    assert_guard_intact(gv_guard, "V workspace")
