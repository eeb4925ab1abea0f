"""Shared helpers of the GPU parity tests: move seeded workload inputs to the
device, run the library, and build the oracle's side from the same inputs.
The oracle side never reads anything the CUDA path produced."""
import numpy as np
import torch

import bit_paged_kv_kv4_gb300 as K
import oracle
from oracle import pool as OP
from workloads import CHUNK, bf16_bits_to_f32, global_scale_from_amax, slots_for

# Parity gate for attention outputs (max-abs error and cosine vs the FP64 oracle).
ATOL = 2e-3
MIN_COS = 0.9999

# Guard bytes after a device buffer: a kernel writing past the buffer's end
# changes them (the whole-buffer compares only see writes inside it).
GUARD_BYTES = 4096
GUARD = 0x5C


def guarded_pool(fmt, num_pages, P, Hkv, D, fill=0):
    """A pool whose device buffer is followed by GUARD_BYTES guard bytes;
    ``pool.buffer`` is the pool itself, ``pool.guard`` the bytes after it."""
    n = K.kv4_pool_bytes(fmt, num_pages, P, Hkv, D)
    raw = torch.empty(n + GUARD_BYTES, dtype=torch.uint8, device="cuda")
    raw[:n].fill_(fill)
    raw[n:].fill_(GUARD)
    pool = K.Pool(fmt, num_pages, P, Hkv, D, buffer=raw)
    pool.buffer, pool.guard = raw[:n], raw[n:]
    return pool


def guarded_empty(shape, fill, dtype=torch.uint8):
    """A uint8 device tensor of `shape` (filled with `fill`) followed by guard
    bytes; returns (tensor, guard)."""
    n = int(np.prod(shape))
    raw = torch.empty(n + GUARD_BYTES, dtype=dtype, device="cuda")
    raw[:n].fill_(fill)
    raw[n:].fill_(GUARD)
    return raw[:n].view(shape), raw[n:]


def assert_guard_intact(guard, what="buffer"):
    torch.cuda.synchronize()
    assert bool((guard == GUARD).all()), f"bytes past the end of the {what} were written"


def dev_bf16(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()


def to_u16(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_close(got, want, atol=ATOL, min_cos=MIN_COS, what=""):
    got = np.asarray(got, np.float64).reshape(-1, want.shape[-1])
    want = np.asarray(want, np.float64).reshape(-1, want.shape[-1])
    err = np.abs(got - want).max()
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err <= atol, f"{what}: max abs error {err:.3g} > {atol}"
    for i in range(want.shape[0]):
        nw, ng = np.linalg.norm(want[i]), np.linalg.norm(got[i])
        if nw == 0:
            assert ng == 0, f"{what}: row {i} should be zero"
            continue
        cos = float(want[i] @ got[i] / (nw * ng))
        assert cos >= min_cos, f"{what}: row {i} cosine {cos:.6f} < {min_cos}"
    return err


class Case:
    """A small explicit decode case: random bf16 K/V for given lengths."""

    def __init__(self, fmt, Hkv, Hq, D, lens, P, seed=0, kv_scale=1.0, outlier_ch=(), spare=2):
        rng = np.random.default_rng(seed)
        self.fmt, self.Hkv, self.Hq, self.D, self.P = fmt, Hkv, Hq, D, P
        self.lens = np.array(lens, np.int32)
        B = len(lens)
        need = [(int(L) + P - 1) // P for L in lens]
        self.num_pages = max(sum(need) + spare, 1)
        perm = np.random.default_rng(seed + 99).permutation(self.num_pages).astype(np.int32)
        mp = max(max(need), 1)
        self.table = np.full((B, mp), -1, np.int32)
        at = 0
        for b, n in enumerate(need):
            self.table[b, :n] = perm[at:at + n]
            at += n
        T = int(sum(lens))
        kf = rng.standard_normal((max(T, 1), Hkv, D)).astype(np.float32) * kv_scale
        vf = rng.standard_normal((max(T, 1), Hkv, D)).astype(np.float32) * kv_scale
        for c in outlier_ch:
            kf[:, :, c] *= 10
            vf[:, :, c] *= 10
        from workloads import f32_to_bf16_bits
        self.k = f32_to_bf16_bits(kf)[:T]
        self.v = f32_to_bf16_bits(vf)[:T]
        self.slots = np.concatenate([slots_for(self.table[b], P, np.arange(L)) for b, L in enumerate(lens)]
                                    + [np.zeros(0, np.int64)]).astype(np.int64)
        amk = np.abs(bf16_bits_to_f32(self.k)).max() if T else 1.0
        amv = np.abs(bf16_bits_to_f32(self.v)).max() if T else 1.0
        if fmt == "fp8":
            from workloads import fp8_scale_from_amax
            self.g = np.array([fp8_scale_from_amax(amk), fp8_scale_from_amax(amv)], np.float32)
        else:
            self.g = np.array([global_scale_from_amax(amk), global_scale_from_amax(amv)], np.float32)
        self.q = f32_to_bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
        self.sm = np.float32(1.0 / np.sqrt(D))

    # oracle side
    def oracle_pool(self, fill=0):
        spec = OP.PoolSpec(self.fmt, self.num_pages, self.P, self.Hkv, self.D)
        pool = OP.new_pool(spec, fill)
        OP.write(pool, spec, self.k, self.v, self.slots, self.g)
        return spec, pool

    def oracle_out(self, rows=None):
        spec, pool = self.oracle_pool()
        return oracle.attention.decode_attention(self.q, pool, spec, self.g, self.table, self.lens,
                                                 self.sm, rows=rows)

    # device side
    def gpu_pool(self, fill=0):
        pool = guarded_pool(self.fmt, self.num_pages, self.P, self.Hkv, self.D, fill)
        self.d_g = torch.from_numpy(self.g).cuda()
        if len(self.slots):
            K.kv4_write(dev_bf16(self.k), dev_bf16(self.v), torch.from_numpy(self.slots).cuda(), pool,
                        self.d_g)
        return pool

    def gpu_out(self, pool, num_splits=0, out_dtype=torch.float32):
        B = len(self.lens)
        S = num_splits
        ws = K.alloc_workspace(B, self.Hq, self.D, S)
        out = torch.full((B, self.Hq, self.D), float("nan"), dtype=out_dtype, device="cuda")
        K.kv4_decode_attention(dev_bf16(self.q), pool, self.d_g, torch.from_numpy(self.table).cuda(),
                               torch.from_numpy(self.lens).cuda(), self.sm, out, num_splits=S,
                               workspace=ws)
        torch.cuda.synchronize()
        return out
