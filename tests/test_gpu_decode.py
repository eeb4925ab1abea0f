"""kv4_decode_attention on the GPU against the FP64 oracle: max-abs error
<= 2e-3 and cosine >= 0.9999 per output row, over NVFP4 and INT4, head dims
64/128/256, GQA groups 1..16, ragged lengths spanning several tiles and
pages, empty and one-token requests, and every split count from one (direct
output) to more splits than tiles."""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
from kv4_testlib import Case, assert_guard_intact, check_close, to_u16
from workloads import TINY

pytestmark = pytest.mark.gpu


def run(c, splits=0, out_dtype=torch.float32):
    pool = c.gpu_pool()
    out = c.gpu_out(pool, num_splits=splits, out_dtype=out_dtype)
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    return out


def test_tiny_workload():
    w = TINY
    L = w.seq_lens()
    c = Case("nvfp4", 1, 2, 64, list(L), 16, seed=0, outlier_ch=(5, 40))
    want = c.oracle_out()
    for S in (1, 2, 4):
        got = run(c, S).cpu().numpy()
        check_close(got, want, what=f"tiny S={S}")


@pytest.mark.parametrize("fmt", ["nvfp4", "int4", "fp8"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_ragged_batch(fmt, D):
    c = Case(fmt, 2, 12, D, [1, 63, 64, 65, 700, 0, 1333], 64 if fmt == "nvfp4" else 48 * 2,
             seed=D, outlier_ch=(1, D - 3))
    want = c.oracle_out()
    for S in (1, 3, 0, 40):
        got = run(c, S).cpu().numpy()
        check_close(got, want, what=f"{fmt} D={D} S={S}")


@pytest.mark.parametrize("G", [1, 2, 6, 8, 11, 16])
def test_gqa_groups(G):
    c = Case("nvfp4", 2, 2 * G, 256, [300, 129], 16, seed=G)
    want = c.oracle_out()
    got = run(c, 2).cpu().numpy()
    check_close(got, want, what=f"G={G}")


def test_int4_large_page():
    c = Case("int4", 2, 16, 256, [1600 * 2 + 77, 900], 1600, seed=3)
    want = c.oracle_out()
    for S in (1, 5):
        check_close(run(c, S).cpu().numpy(), want, what=f"int4 P1600 S={S}")


def test_bf16_output_within_one_ulp():
    c = Case("nvfp4", 1, 6, 256, [500, 77], 64, seed=4)
    want = c.oracle_out()
    got = run(c, 3, torch.bfloat16).float().cpu().numpy()
    want_b = torch.from_numpy(want).to(torch.bfloat16).float().numpy()
    ulp = np.abs(want_b) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - want_b) <= ulp * 1.01 + 2e-3)


def test_deterministic_and_split_consistent():
    c = Case("nvfp4", 2, 12, 256, [5000, 2222], 64, seed=6)
    pool = c.gpu_pool()
    a = c.gpu_out(pool, 7).cpu().numpy()
    b = c.gpu_out(pool, 7).cpu().numpy()
    assert np.array_equal(a, b)
    d = c.gpu_out(pool, 1).cpu().numpy()
    assert np.abs(a - d).max() < 1e-4


def test_large_query_prescaled():
    # |q| far beyond the f16 range is pre-scaled by a power of two in the
    # kernel; unit-scale K/V, so the gate applies as it stands
    c = Case("nvfp4", 1, 4, 128, [200], 32, seed=7)
    from workloads import f32_to_bf16_bits, bf16_bits_to_f32
    c.q = f32_to_bf16_bits(bf16_bits_to_f32(c.q) * np.float32(1e5))
    c.sm = np.float32(1e-9)
    want = c.oracle_out()
    check_close(run(c, 2).cpu().numpy(), want, what="large |q|")


def test_large_kv_magnitudes():
    # K and V 300 times larger (global scales follow); the output inherits
    # V's scale, so the gate applies to out / 300 (the unit-scale output)
    c = Case("nvfp4", 1, 4, 128, [200], 32, seed=7, kv_scale=300.0)
    want = c.oracle_out()
    check_close(run(c, 2).cpu().numpy() / 300.0, want / 300.0, what="K, V x300")


def test_bad_block_table_entry_is_flagged_not_faulted():
    c = Case("nvfp4", 1, 2, 64, [100], 16, seed=8)
    pool = c.gpu_pool()
    c.table = c.table.copy()
    c.table[0, 2] = c.num_pages + 5
    K.kv4_device_error()
    out = c.gpu_out(pool, 2)
    assert K.kv4_device_error() == 4
    c.lens = np.array([c.table.shape[1] * 16 + 1], np.int32)   # beyond the table
    c.table[0, 2] = 0
    out = c.gpu_out(pool, 1)
    assert K.kv4_device_error() == 4


@pytest.mark.parametrize("G", [1, 6, 8, 11])
def test_fp8_gqa_groups_and_pages(G):
    """FP8 comparison format: GQA groups, pages that 32 does not divide, splits."""
    c = Case("fp8", 2, 2 * G, 256, [300, 129, 16], 48, seed=100 + G, outlier_ch=(7,))
    want = c.oracle_out()
    for S in (0, 1, 5):
        check_close(run(c, S).cpu().numpy(), want, what=f"fp8 G={G} S={S}")
