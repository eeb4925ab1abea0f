"""Host-side logic with no GPU: the decode-source hash that keys recorded
ncu traffic, the FP8 input generator, and the k8v4 workspace sizing."""
import numpy as np
import torch

import bench
import workloads as W


def test_decode_hash_ignores_comments_and_blank_space(tmp_path, monkeypatch):
    src = tmp_path / "bit_paged_kv_kv4_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "kv4_decode.cu").write_text("int f(int x) { return x + 1; }  // one\n/* block */\n")
    (src / "kv4_decode4.cu").write_text("int g(int x) { return x; }\n")
    (src / "kv4_device.cuh").write_text("#pragma once\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.decode_source_hash()
    (src / "kv4_decode.cu").write_text("int f(int x) {\n  return x + 1;  // two\n}\n")
    assert bench.decode_source_hash() == h0                 # comments and layout only
    (src / "kv4_decode.cu").write_text("int f(int x) { return x + 2; }\n")
    h1 = bench.decode_source_hash()
    assert h1 != h0                                         # code changed
    (src / "kv4_decode4.cu").write_text("int g(int x) { return -x; }\n")
    assert bench.decode_source_hash() != h1                 # either kernel file counts


def test_fp8_kv_codes_saturate_and_repeat():
    a, s = W.fp8_kv_codes(3, 50, 2, 64, "cpu", [[1], [7]], 30.0)
    b, _ = W.fp8_kv_codes(3, 50, 2, 64, "cpu", [[1], [7]], 30.0)
    assert torch.equal(a, b)                                 # seeded
    assert a.dtype == torch.uint8 and a.shape == (2, 50, 2, 64)
    codes = a.numpy()
    assert not np.any((codes & 0x7F) == 0x7F)                # no NaN code
    # scales from the draws' maxima: the largest magnitude encodes to 448
    assert np.any((codes & 0x7F) == 0x7E)
    # fixed scales smaller than the data saturate instead of producing NaN
    c, _ = W.fp8_kv_codes(4, 50, 2, 64, "cpu", scales=np.array([1e-3, 1e-3], np.float32))
    assert not np.any((c.numpy() & 0x7F) == 0x7F)


def _a256(x):
    return (x + 255) // 256 * 256


def test_k8v4_workspace_sizing():
    """The k8v4 decode workspace has the layout of kv4_decode_attention's:
    tile offsets [B+1] int64, then per slot 8 piece states of 16 bytes and 8
    piece rows of D floats; slots = R + B*Hkv*S, R the device's resident CTAs
    (a wave of persistent CTAs, one piece each at most per unit)."""
    import bit_paged_kv_kv4_gb300 as K
    B, Hkv, D = 16, 4, 256

    def size(R, S):
        slots = R + B * Hkv * S
        return _a256((B + 1) * 8) + _a256(slots * 8 * 16) + slots * 8 * D * 4

    n19 = K.kv4_k8v4_workspace_bytes(B, Hkv, D, 19)
    R = next(r for r in range(1, 100000) if size(r, 19) >= n19)
    assert size(R, 19) == n19
    assert K.kv4_k8v4_workspace_bytes(B, Hkv, D, 20) == size(R, 20)
    assert K.kv4_k8v4_workspace_bytes(B, Hkv, 64, 1) == _a256((B + 1) * 8) + _a256((R + B * Hkv) * 128) + (R + B * Hkv) * 8 * 64 * 4
    assert K.kv4_k8v4_workspace_bytes(2, 2, 64, 0) == 0     # no split count: nothing to size
