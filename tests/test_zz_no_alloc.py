"""kv4_decode_attention_static_ws: the decode entry point for callers that
cannot allocate device memory (a framework that owns all device allocations,
or a loop that cannot take an allocation's synchronisation).  Its split
scratch is the library's fixed 8 MiB device array instead of a caller
workspace.

Checked through the C ABI on a GPU: two calls in a row give bitwise the
output of the regular entry point with the same split count, and both stay
within the decode parity gate of the FP64 oracle; a request too large for
the array is refused without a launch, and an invalid argument gets the
regular entry point's own message.  This file is collected last on purpose,
and also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
from kv4_testlib import ATOL, Case, check_close, dev_bf16

pytestmark = pytest.mark.gpu


def _static_call(lib, c, pool, q, table, lens, out, splits):
    return lib.kv4_decode_attention_static_ws(
        ctypes.c_void_p(q.data_ptr()), pool.ref, ctypes.c_void_p(c.d_g.data_ptr()),
        ctypes.c_void_p(table.data_ptr()), table.shape[1], ctypes.c_void_p(lens.data_ptr()),
        len(c.lens), c.Hq, float(c.sm), splits, ctypes.c_void_p(out.data_ptr()), 1,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
def test_static_workspace_matches_regular_entry_point_twice(fmt):
    lib = K.load(build_if_missing=True)
    c = Case(fmt, 2, 12, 256, [3000, 77, 1, 1500], 64, seed=21, outlier_ch=(5,))
    pool = c.gpu_pool()
    S = 9
    ref = c.gpu_out(pool, num_splits=S).cpu().numpy()
    want = c.oracle_out()
    q = dev_bf16(c.q)
    table = torch.from_numpy(c.table).cuda()
    lens = torch.from_numpy(c.lens).cuda()
    for call in range(2):
        out = torch.full((len(c.lens), c.Hq, c.D), float("nan"), device="cuda")
        st = _static_call(lib, c, pool, q, table, lens, out, S)
        assert st == 0, lib.kv4_last_error_message().decode()
        torch.cuda.synchronize()
        assert K.kv4_device_error() == 0
        got = out.cpu().numpy()
        assert np.array_equal(got, ref), f"static workspace, call {call + 1}: not bitwise equal"
        check_close(got, want, atol=ATOL, what=f"static workspace vs oracle, call {call + 1}")


def test_static_workspace_refuses_oversized_requests():
    lib = K.load(build_if_missing=True)
    c = Case("nvfp4", 1, 8, 256, [64] * 8, 64, seed=22)
    pool = c.gpu_pool()
    # 8 requests x 8 heads x 1024 splits x (256 + 4) floats is far above 8 MiB
    out = torch.zeros((8, 8, 256), device="cuda")
    table = torch.from_numpy(c.table).cuda()
    lens = torch.from_numpy(c.lens).cuda()
    st = _static_call(lib, c, pool, dev_bf16(c.q), table, lens, out, 1024)
    assert st == 1
    msg = lib.kv4_last_error_message().decode()
    assert "8388608" in msg and "static workspace" in msg
    torch.cuda.synchronize()
    assert float(out.abs().sum()) == 0.0                # nothing was launched


def test_static_workspace_reports_argument_errors_first():
    lib = K.load(build_if_missing=True)
    c = Case("nvfp4", 2, 6, 256, [64] * 4, 64, seed=23)
    pool = c.gpu_pool()
    table = torch.from_numpy(c.table).cuda()
    lens = torch.from_numpy(c.lens).cuda()
    out = torch.zeros((4, 6, 256), device="cuda")
    # 7 query heads over 2 kv heads, with a split count whose scratch would
    # not fit either: the argument error is the one reported
    st = lib.kv4_decode_attention_static_ws(
        ctypes.c_void_p(dev_bf16(c.q).data_ptr()), pool.ref, ctypes.c_void_p(c.d_g.data_ptr()),
        ctypes.c_void_p(table.data_ptr()), table.shape[1], ctypes.c_void_p(lens.data_ptr()),
        4, 7, float(c.sm), 1024, ctypes.c_void_p(out.data_ptr()), 1,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 1
    msg = lib.kv4_last_error_message().decode()
    assert "multiple of num_kv_heads" in msg and "static workspace" not in msg
