"""The C ABI without a GPU: the library builds and loads, exports every
function include/kv4.h declares, and rejects bad arguments on the host
before any CUDA call (the validation contract of the header)."""
import ctypes
import os
import re

import pytest

import bit_paged_kv_kv4_gb300 as K
from bit_paged_kv_kv4_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kv4.h")


@pytest.fixture(scope="module")
def lib():
    return K.load(build_if_missing=True)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("kv4_write", "kv4_decode_attention", "kv4_dequant_prefix", "kv4_extend_attention",
              "kv4_calibrate_global_scale"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def desc(fmt=0, pages=4, P=64, H=2, D=256, base=None):
    return K._PoolDesc(fmt, pages, P, H, D, 0, base)


def test_pool_sizes(lib):
    d = desc()
    assert lib.kv4_pool_chunk_bytes(ctypes.byref(d)) == 64 * 288
    assert lib.kv4_pool_bytes(ctypes.byref(d)) == 4 * 2 * 64 * 288
    assert lib.kv4_pool_chunk_bytes(ctypes.byref(desc(fmt=1, P=1600))) == 422400
    assert lib.kv4_pool_chunk_bytes(ctypes.byref(desc(fmt=2))) == 64 * 2 * 256      # FP8: 16 B per 16 values
    for bad in (desc(P=8), desc(P=40), desc(D=96), desc(H=0), desc(pages=0), desc(fmt=7)):
        assert lib.kv4_pool_bytes(ctypes.byref(bad)) == 0


def test_workspace_sizes(lib):
    assert lib.kv4_decode_workspace_bytes(2, 8, 256, 1) == 0          # direct output
    a0 = lib.kv4_decode_workspace_bytes(2, 8, 256, 0)
    a5 = lib.kv4_decode_workspace_bytes(2, 8, 256, 5)
    assert 0 < a0 < a5
    # slots grow by one per (request, head, split): 16 heads x 4 more splits
    assert a5 - a0 == 2 * 8 * 4 * 8 * (16 + 256 * 4)
    assert lib.kv4_decode_workspace_bytes(0, 8, 256, 0) == 0


def _status(lib, st):
    return st, lib.kv4_last_error_message().decode()


def test_host_validation_rejects_without_gpu(lib):
    d = desc(base=1 << 20)
    p = ctypes.byref(d)
    fake = ctypes.c_void_p(1 << 20)
    # fmt mismatch
    st, msg = _status(lib, lib.kv4_write(fake, fake, fake, 4, p, fake, 1, None))
    assert st == 1 and "fmt" in msg
    # unaligned k
    st, _ = _status(lib, lib.kv4_write(ctypes.c_void_p((1 << 20) + 2), fake, fake, 4, p, fake, 0, None))
    assert st == 1
    # NVFP4 without global scale
    st, msg = _status(lib, lib.kv4_write(fake, fake, fake, 4, p, None, 0, None))
    assert st == 1 and "global" in msg
    # zero tokens is a no-op
    assert lib.kv4_write(None, None, None, 0, p, None, 0, None) == 0
    # unsupported head_dim
    d96 = desc(D=96, base=1 << 20)
    assert lib.kv4_write(fake, fake, fake, 4, ctypes.byref(d96), fake, 0, None) == 2
    # unaligned pool base
    dmis = desc(base=(1 << 20) + 128)
    assert lib.kv4_write(fake, fake, fake, 4, ctypes.byref(dmis), fake, 0, None) == 1
    # decode: bad splits, bad head ratio, missing workspace
    args = lambda **kw: dict(dict(q=fake, pool=p, g=fake, bt=fake, mp=8, sl=fake, B=2, Hq=12,
                                  sm=0.0625, S=4, ws=None, wsb=0, out=fake, f32=1), **kw)

    def dec(a):
        return lib.kv4_decode_attention(a["q"], a["pool"], a["g"], a["bt"], a["mp"], a["sl"], a["B"],
                                        a["Hq"], a["sm"], a["S"], a["ws"], a["wsb"], a["out"],
                                        a["f32"], None)
    assert dec(args(S=-1)) == 1
    assert dec(args(S=2000)) == 1
    assert dec(args(Hq=7)) == 1
    assert dec(args(sm=float("nan"))) == 1
    st, msg = _status(lib, dec(args()))
    assert st == 1 and "workspace" in msg
    assert dec(args(B=0)) == 0
    # prefix: max_prefix_len beyond the table
    assert lib.kv4_dequant_prefix(p, fake, fake, 2, fake, fake, 1, 1000, fake, fake, fake, None) == 1
    assert lib.kv4_dequant_prefix(p, fake, fake, 2, fake, fake, 1, 0, fake, fake, fake, None) == 0
    # FP8 pools: write and decode need the per-tensor scales; no prefix dequant
    d8 = desc(fmt=2, base=1 << 20)
    st, msg = _status(lib, lib.kv4_write(fake, fake, fake, 4, ctypes.byref(d8), None, 2, None))
    assert st == 1 and "scale" in msg
    st, msg = _status(lib, lib.kv4_dequant_prefix(ctypes.byref(d8), fake, fake, 2, fake, fake, 1, 1,
                                                  fake, fake, fake, None))
    assert st == 2 and "FP8" in msg
    # calibration: output pointer, head_dim, alignment
    assert lib.kv4_calibrate_global_scale(fake, fake, 4, 2, 256, None, None) == 1
    assert lib.kv4_calibrate_global_scale(fake, fake, 4, 2, 96, fake, None) == 2
    assert lib.kv4_calibrate_global_scale(ctypes.c_void_p((1 << 20) + 2), fake, 4, 2, 256, fake, None) == 1


def test_status_strings(lib):
    for s in range(6):
        assert lib.kv4_status_str(s).decode().startswith("KV4_")


def test_build_is_in_tree():
    assert os.path.dirname(_build.LIB) == os.path.dirname(K.__file__)


def test_extend_validation_without_gpu(lib):
    fake = ctypes.c_void_p(1 << 20)

    def ext(**kw):
        a = dict(q=fake, ck=fake, cv=fake, pk=fake, pv=fake, s=fake, pl=fake, cp=fake, cl=fake,
                 cc=fake, B=2, mc=300, Hq=24, Hkv=4, D=256, sm=0.0625, out=fake, f32=0)
        a.update(kw)
        return lib.kv4_extend_attention(a["q"], a["ck"], a["cv"], a["pk"], a["pv"], a["s"], a["pl"],
                                        a["cp"], a["cl"], a["cc"], a["B"], a["mc"], a["Hq"], a["Hkv"],
                                        a["D"], a["sm"], a.get("ws"), a.get("wsb", 0), a["out"], a["f32"],
                                        None)
    assert ext(Hq=25) == 1                      # heads not a multiple of kv heads
    assert ext(D=96) == 2                       # head_dim not built
    assert ext(sm=0.0) == 1 and ext(sm=float("nan")) == 1
    assert ext(B=-1) == 1 and ext(mc=-5) == 1
    assert ext(B=70000) == 1
    assert ext(pk=None) == 1                    # missing prefix workspace
    st, msg = _status(lib, ext(q=ctypes.c_void_p((1 << 20) + 8)))
    assert st == 1 and "aligned" in msg
    assert ext(B=0) == 0 and ext(mc=0) == 0     # nothing to do


def test_write_fp8_validation_without_gpu(lib):
    d = desc(base=1 << 20)
    p = ctypes.byref(d)
    fake = ctypes.c_void_p(1 << 20)
    st, msg = _status(lib, lib.kv4_write_fp8(fake, fake, None, fake, 4, p, fake, 0, None))
    assert st == 1 and "in_scale" in msg                    # FP8 input without its scales
    assert lib.kv4_write_fp8(fake, fake, fake, fake, 4, p, fake, 1, None) == 1   # fmt mismatch
    assert lib.kv4_write_fp8(None, None, None, None, 0, p, None, 0, None) == 0   # nothing to do


def test_k8v4_validation_without_gpu(lib):
    fake = ctypes.c_void_p(1 << 20)
    d = desc(fmt=3, base=1 << 20)
    p = ctypes.byref(d)
    assert lib.kv4_pool_chunk_bytes(p) == 64 * (256 + 128 + 4)
    # the generic entry points refuse a k8v4 pool
    assert lib.kv4_write(fake, fake, fake, 4, p, fake, 3, None) == 2
    assert lib.kv4_dequant_prefix(p, fake, fake, 2, fake, fake, 1, 1, fake, fake, fake, None) == 2
    assert lib.kv4_decode_attention(fake, p, fake, fake, 8, fake, 2, 8, 0.0625, 4, fake, 1 << 20,
                                    fake, 1, None) == 2
    # k8v4 entries: scale pointer, head ratio, group size, workspace size
    assert lib.kv4_k8v4_write(fake, fake, fake, 4, p, None, None) == 1
    assert lib.kv4_k8v4_write(fake, fake, fake, 0, p, None, None) == 0
    dec = lambda **kw: lib.kv4_k8v4_decode_attention(
        fake, p, fake, fake, 8, fake, kw.get("B", 2), kw.get("Hq", 8), 0.0625, kw.get("S", 4), fake,
        kw.get("ws", 1 << 30), fake, 1, None)
    assert dec(Hq=7) == 1 and dec(Hq=18) == 2 and dec(S=0) == 1
    assert dec(ws=16) == 1
    assert lib.kv4_k8v4_workspace_bytes(2, 2, 256, 4) > 2 * 2 * 4 * 8 * 256 * 4
    nv = desc(fmt=0, base=1 << 20)
    assert lib.kv4_k8v4_write(fake, fake, fake, 4, ctypes.byref(nv), fake, None) == 1


def test_every_declared_function_has_a_binding_signature():
    """The binding declares argument and result types for every C entry point
    of the header (an undeclared one would be called with ctypes' defaults)."""
    import inspect
    src = inspect.getsource(K._load)
    for name in declared_functions():
        assert f'"{name}"' in src, name


def test_extend_workspace_sizing_and_checks(lib):
    """The extend workspace holds one partial state (128 rows of D floats and
    two floats) per piece of the split items: at most one piece per SM, and
    nothing when the items fill whole waves."""
    sms = 152   # no device here: the library assumes 152 SMs
    n = lib.kv4_extend_workspace_bytes(1, 8192, 24, 256)      # 1536 items = 10 x 152 + 16
    pieces = 16 * (152 // 16)
    assert n == (pieces * 128 * 256 * 4 + 255) // 256 * 256 + pieces * 128 * 8
    assert lib.kv4_extend_workspace_bytes(1, 128 * 152, 1, 64) == 0     # whole waves: no split
    assert lib.kv4_extend_workspace_bytes(1, 128, 100, 64) == 0         # 100 items: 152 // 100 < 2
    assert lib.kv4_extend_workspace_bytes(1, 128, 24, 256) > 0          # 24 items in 6 pieces each
    assert lib.kv4_extend_workspace_bytes(0, 128, 24, 256) == 0
    assert n <= sms * 128 * (256 * 4 + 8) + 256
    fake = ctypes.c_void_p(1 << 20)
    st = lib.kv4_extend_attention(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 8192, 24,
                                  4, 256, 0.0625, fake, n - 1, fake, 0, None)
    assert st == 1                               # workspace too small


def test_decode_step_validation_without_gpu(lib):
    """kv4_decode_step: NVFP4 / INT4 pools with at most 8 query heads per kv
    head, non-NULL 16-byte aligned new K/V; everything else is refused before
    any CUDA call."""
    fake = ctypes.c_void_p(1 << 20)

    def step(d, k=fake, v=fake, Hq=8):
        return _status(lib, lib.kv4_decode_step(fake, k, v, ctypes.byref(d), fake, fake, 8, fake, 2, Hq,
                                                0.0625, 1, None, 0, fake, 1, None))
    d = desc(base=1 << 20)                 # NVFP4
    st, msg = step(desc(fmt=2, base=1 << 20))
    assert st == 2 and "NVFP4 and INT4" in msg
    Hkv = d.num_kv_heads
    st, msg = step(d, Hq=16 * Hkv)
    assert st == 2 and "8 query heads" in msg
    st, msg = step(d, k=None)
    assert st == 1 and "k_new" in msg
    st, msg = step(d, v=ctypes.c_void_p((1 << 20) + 2))
    assert st == 1 and "aligned" in msg
