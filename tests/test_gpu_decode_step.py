"""kv4_decode_step (the step's new token written by the decode kernel itself)
against the two calls it stands for, kv4_write of each request's last token
and then kv4_decode_attention: the pool bytes and the output must be bitwise
the same.  One case is also held to the FP64 oracle's gate."""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
from kv4_testlib import ATOL, Case, assert_guard_intact, check_close, dev_bf16, guarded_pool

pytestmark = pytest.mark.gpu


def _split(c):
    """Slots of every token but each request's last, and the last tokens'
    K/V ([B, Hkv, D]) with their slots."""
    starts = np.concatenate([[0], np.cumsum(c.lens)])[:-1]
    last = [int(s + L - 1) for s, L in zip(starts, c.lens) if L > 0]
    keep = np.ones(len(c.slots), bool)
    keep[last] = False
    B = len(c.lens)
    k_new = np.zeros((B, c.Hkv, c.D), np.uint16)
    v_new = np.zeros((B, c.Hkv, c.D), np.uint16)
    slot_new = np.full(B, -1, np.int64)
    for b, (s, L) in enumerate(zip(starts, c.lens)):
        if L > 0:
            k_new[b], v_new[b], slot_new[b] = c.k[s + L - 1], c.v[s + L - 1], c.slots[s + L - 1]
    return keep, k_new, v_new, slot_new


def _pools(c, keep, fill):
    pools = []
    c.d_g = torch.from_numpy(c.g).cuda()
    for _ in range(2):
        pool = guarded_pool(c.fmt, c.num_pages, c.P, c.Hkv, c.D, fill)
        if keep.any():
            K.kv4_write(dev_bf16(c.k[keep]), dev_bf16(c.v[keep]), torch.from_numpy(c.slots[keep]).cuda(), pool,
                        c.d_g)
        pools.append(pool)
    return pools


def run_both(c, num_splits, fill=0x5A, out_dtype=torch.float32):
    keep, k_new, v_new, slot_new = _split(c)
    p_ref, p_step = _pools(c, keep, fill)
    B = len(c.lens)
    table = torch.from_numpy(c.table).cuda()
    lens = torch.from_numpy(c.lens).cuda()
    q = dev_bf16(c.q)
    ws = K.alloc_workspace(B, c.Hq, c.D, num_splits)
    out_ref = torch.full((B, c.Hq, c.D), float("nan"), dtype=out_dtype, device="cuda")
    out_step = torch.full_like(out_ref, float("nan"))
    # the two calls: the new tokens' write, then the decode
    K.kv4_write(dev_bf16(k_new), dev_bf16(v_new), torch.from_numpy(slot_new).cuda(), p_ref, c.d_g)
    K.kv4_decode_attention(q, p_ref, c.d_g, table, lens, c.sm, out_ref, num_splits=num_splits, workspace=ws)
    # one call
    K.kv4_decode_step(q, dev_bf16(k_new), dev_bf16(v_new), p_step, c.d_g, table, lens, c.sm, out_step,
                      num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert_guard_intact(p_step.guard, "pool")
    a, b = p_ref.buffer.cpu().numpy(), p_step.buffer.cpu().numpy()
    diff = np.nonzero(a != b)[0]
    assert diff.size == 0, f"{diff.size} pool bytes differ, first at {diff[:8]}"
    assert torch.equal(out_ref, out_step)
    return out_step


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
@pytest.mark.parametrize("D,P", [(64, 16), (128, 32), (256, 64)])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_step_equals_write_then_decode(fmt, D, P, num_splits):
    # last positions at an even and an odd offset of a page (NVFP4 V shares a
    # pair row with the token before or after), at a page's last slot, the
    # first token of a request, and an empty request
    lens = [P * 3 + 5, P * 2, 1, 2 * P + 2, 0, 37]
    c = Case(fmt, 2, 8, D, lens, P, seed=D + P + num_splits)
    run_both(c, num_splits)


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
def test_decode_step_long_requests_and_gqa(fmt):
    # many tiles per unit (the last tile owned by one CTA of the balanced
    # schedule), query groups of 6 and 1
    for Hkv, Hq in ((4, 24), (4, 4)):
        c = Case(fmt, Hkv, Hq, 256, [3000, 1777, 64], 64, seed=Hq)
        run_both(c, 0)


def test_decode_step_against_the_oracle():
    c = Case("nvfp4", 2, 8, 128, [300, 45, 129], 32, seed=9, outlier_ch=(3, 50))
    out = run_both(c, 0).cpu().numpy()
    check_close(out, c.oracle_out(), atol=ATOL, what="decode step vs oracle")


def test_decode_step_refuses_fp8_and_large_groups():
    c = Case("fp8", 2, 8, 128, [40, 10], 16, seed=1)
    pool = c.gpu_pool()
    kn = torch.zeros((2, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((2, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(K.Kv4Error):
        K.kv4_decode_step(dev_bf16(c.q), kn, kn, pool, c.d_g, torch.from_numpy(c.table).cuda(),
                          torch.from_numpy(c.lens).cuda(), c.sm, out, num_splits=1)


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
def test_decode_step_more_requests_than_a_cta_has_threads(fmt):
    # 150 requests: the balanced schedule finds the new-token jobs by its
    # general scan (rounds over request blocks); then one CTA per unit
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, 70, 150)]
    c = Case(fmt, 2, 4, 128, lens, 16, seed=11)
    run_both(c, 0)
    run_both(c, 1)


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
def test_decode_step_bf16_output(fmt):
    c = Case(fmt, 2, 8, 128, [200, 31, 64], 32, seed=21)
    # bitwise equal to the two calls' bf16 output (whose rounding the decode
    # tests hold to one bf16 ulp of the FP32 result)
    out = run_both(c, 0, out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16 and torch.isfinite(out.float()).all()
