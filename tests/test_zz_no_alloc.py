"""kv4_decode_attention_static_ws: the decode entry point for callers that
cannot allocate device memory (a framework that owns all device allocations,
or a loop that cannot take an allocation's synchronisation).  Its split
scratch is the library's fixed 8 MiB device array instead of a caller
workspace.

Checked through the C ABI on a GPU: two calls in a row match the regular
entry point (same split count) within the parity tolerance of the other
decode tests, and a request too large for the array is refused without a
launch.  This file is collected last on purpose, and also passes on its own.
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
        check_close(got, ref, atol=ATOL, what=f"static workspace, call {call + 1}")


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
