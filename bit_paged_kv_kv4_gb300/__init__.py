"""Python binding of libkv4 (include/kv4.h): a 4-bit paged KV cache for GB300.

Argument marshalling only.  Every step of the write, decode, prefix, extend
and calibration paths runs in the library's CUDA kernels; torch supplies
device memory and streams.
There is no fallback: if libkv4.so is missing or cannot load, importing the
binding's functions raises.

The functions carry the C names: ``kv4_write``, ``kv4_decode_attention``,
``kv4_dequant_prefix``, ``kv4_extend_attention``,
``kv4_calibrate_global_scale``, plus the sizing helpers and ``Pool`` (the
pool descriptor with its device buffer).
"""
import ctypes
import os

import torch

from . import _build

KV4_NVFP4 = 0
KV4_INT4_PTH = 1
KV4_FP8 = 2
KV4_K8V4 = 3
FMT = {"nvfp4": KV4_NVFP4, "int4": KV4_INT4_PTH, "fp8": KV4_FP8, "k8v4": KV4_K8V4}

_lib = None


class Kv4Error(RuntimeError):
    def __init__(self, status, where):
        msg = _load().kv4_last_error_message().decode()
        super().__init__(f"{where}: {_load().kv4_status_str(status).decode()} {msg}".strip())
        self.status = status


class _PoolDesc(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("base", ctypes.c_void_p)]


def library_path():
    return _build.LIB


def _load(build_if_missing=False):
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libkv4 is not built ({path}); run bit_paged_kv_kv4_gb300._build.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(_PoolDesc)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sig = {
        "kv4_pool_chunk_bytes": (i64, [P]),
        "kv4_pool_bytes": (i64, [P]),
        "kv4_write": (i32, [vp, vp, vp, i64, P, vp, i32, vp]),
        "kv4_write_fp8": (i32, [vp, vp, vp, vp, i64, P, vp, i32, vp]),
        "kv4_decode_workspace_bytes": (i64, [i32, i32, i32, i32]),
        "kv4_decode_attention": (i32, [vp, P, vp, vp, i32, vp, i32, i32, f32, i32, vp, i64, vp,
                                       i32, vp]),
        "kv4_decode_step": (i32, [vp, vp, vp, P, vp, vp, i32, vp, i32, i32, f32, i32, vp, i64, vp,
                                  i32, vp]),
        "kv4_dequant_prefix": (i32, [P, vp, vp, i32, vp, vp, i32, i32, vp, vp, vp, vp]),
        "kv4_calibrate_global_scale": (i32, [vp, vp, i64, i32, i32, vp, vp]),
        "kv4_extend_workspace_bytes": (i64, [i32, i32, i32, i32]),
        "kv4_extend_attention": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                       i32, i32, f32, vp, i64, vp, i32, vp]),
        "kv4_decode_attention_static_ws": (i32, [vp, P, vp, vp, i32, vp, i32, i32, f32, i32, vp,
                                                 i32, vp]),
        "kv4_k8v4_write": (i32, [vp, vp, vp, i64, P, vp, vp]),
        "kv4_k8v4_workspace_bytes": (i64, [i32, i32, i32, i32]),
        "kv4_k8v4_decode_attention": (i32, [vp, P, vp, vp, i32, vp, i32, i32, f32, i32, vp, i64, vp,
                                            i32, vp]),
        "kv4_device_error": (i32, []),
        "kv4_status_str": (ctypes.c_char_p, [i32]),
        "kv4_last_error_message": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def load(build_if_missing=False):
    """Load libkv4.so (optionally building it first); returns the ctypes CDLL."""
    return _load(build_if_missing)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != 0:
        raise Kv4Error(status, where)


class Pool:
    """One layer's paged pool: the C descriptor plus its device buffer.

    ``buffer`` is a uint8 CUDA tensor of ``nbytes`` bytes (256-byte aligned);
    pass ``device=None`` to describe a pool without allocating (sizing only).
    """

    def __init__(self, fmt, num_pages, page_size, num_kv_heads, head_dim, device="cuda",
                 buffer=None):
        self.fmt = FMT[fmt] if isinstance(fmt, str) else int(fmt)
        self.desc = _PoolDesc(self.fmt, num_pages, page_size, num_kv_heads, head_dim, 0, None)
        self.nbytes = _load().kv4_pool_bytes(ctypes.byref(self.desc))
        if self.nbytes == 0:
            raise ValueError("invalid pool shape")
        self.chunk_bytes = _load().kv4_pool_chunk_bytes(ctypes.byref(self.desc))
        if buffer is None and device is not None:
            buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        if buffer is not None:
            if buffer.numel() < self.nbytes or buffer.data_ptr() % 256:
                raise ValueError("pool buffer too small or not 256-byte aligned")
            self.desc.base = buffer.data_ptr()
        self.buffer = buffer
        self.num_pages, self.page_size = num_pages, page_size
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim

    @property
    def ref(self):
        return ctypes.byref(self.desc)


def kv4_pool_bytes(fmt, num_pages, page_size, num_kv_heads, head_dim):
    d = _PoolDesc(FMT[fmt] if isinstance(fmt, str) else fmt, num_pages, page_size, num_kv_heads,
                  head_dim, 0, None)
    return _load().kv4_pool_bytes(ctypes.byref(d))


def kv4_write(k, v, slot_mapping, pool, layer_global_scale, fmt=None, stream=None):
    """Quantise bf16 k, v [T, Hkv, D] into ``pool`` at ``slot_mapping`` (int64 [T])."""
    fmt = pool.fmt if fmt is None else (FMT[fmt] if isinstance(fmt, str) else fmt)
    st = _load().kv4_write(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0], pool.ref,
                           _ptr(layer_global_scale), fmt, _stream(stream))
    _check(st, "kv4_write")


def kv4_write_fp8(k, v, in_scale, slot_mapping, pool, layer_global_scale, fmt=None, stream=None):
    """Quantise FP8 E4M3 k, v (uint8 [T, Hkv, D], per-tensor scales in_scale
    float32 [2]) into ``pool`` at ``slot_mapping``."""
    fmt = pool.fmt if fmt is None else (FMT[fmt] if isinstance(fmt, str) else fmt)
    st = _load().kv4_write_fp8(_ptr(k), _ptr(v), _ptr(in_scale), _ptr(slot_mapping), k.shape[0],
                               pool.ref, _ptr(layer_global_scale), fmt, _stream(stream))
    _check(st, "kv4_write_fp8")


def kv4_decode_workspace_bytes(batch, num_q_heads, head_dim, num_splits):
    return _load().kv4_decode_workspace_bytes(batch, num_q_heads, head_dim, num_splits)


def kv4_decode_attention(q, pool, layer_global_scale, block_table, seq_lens, sm_scale,
                         out, num_splits=0, workspace=None, stream=None):
    """Decode attention of q [B, Hq, D] (bf16) over ``pool`` into ``out``
    ([B, Hq, D], float32 or bf16).  ``workspace``: uint8 CUDA tensor of at
    least kv4_decode_workspace_bytes(...) bytes when more than one split."""
    B, Hq, D = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _load().kv4_decode_attention(
        _ptr(q), pool.ref, _ptr(layer_global_scale), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), B, Hq, float(sm_scale), int(num_splits), _ptr(workspace), ws_bytes,
        _ptr(out), 1 if out.dtype == torch.float32 else 0, _stream(stream))
    _check(st, "kv4_decode_attention")


def kv4_decode_step(q, k_new, v_new, pool, layer_global_scale, block_table, seq_lens, sm_scale,
                    out, num_splits=0, workspace=None, stream=None):
    """One decode step in one kernel: each request's new token (k_new, v_new
    [B, Hkv, D] bf16) written into position seq_lens[b] - 1 of its pages,
    then decode attention as kv4_decode_attention (same arguments)."""
    B, Hq, D = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _load().kv4_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), pool.ref, _ptr(layer_global_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, Hq, float(sm_scale), int(num_splits), _ptr(workspace),
        ws_bytes, _ptr(out), 1 if out.dtype == torch.float32 else 0, _stream(stream))
    _check(st, "kv4_decode_step")


def kv4_decode_attention_static_ws(q, pool, layer_global_scale, block_table, seq_lens, sm_scale,
                                   out, num_splits=0, stream=None):
    """kv4_decode_attention without a caller workspace, for callers that cannot
    allocate device memory: the split scratch is the library's fixed 8 MiB
    device array, shared by every call (serialise calls on the GPU)."""
    B, Hq, D = q.shape
    st = _load().kv4_decode_attention_static_ws(
        _ptr(q), pool.ref, _ptr(layer_global_scale), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), B, Hq, float(sm_scale), int(num_splits), _ptr(out),
        1 if out.dtype == torch.float32 else 0, _stream(stream))
    _check(st, "kv4_decode_attention_static_ws")


def kv4_calibrate_global_scale(k, v, out, stream=None):
    """NVFP4 global scales {g_K, g_V} of bf16 k, v [T, Hkv, D] into ``out``
    (float32 CUDA tensor of 2): amax / 2688 each, 1 for an all-zero tensor."""
    T, H, D = k.shape
    st = _load().kv4_calibrate_global_scale(_ptr(k), _ptr(v), T, H, D, _ptr(out), _stream(stream))
    _check(st, "kv4_calibrate_global_scale")


def kv4_dequant_prefix(pool, layer_global_scale, block_table, prefix_lens, cu_prefix,
                       max_prefix_len, fp8_scale, fp8_k, fp8_v, stream=None):
    """Dequantise each request's cached prefix into E4M3 workspaces
    fp8_k / fp8_v (uint8 [sum prefix_lens, Hkv, D])."""
    st = _load().kv4_dequant_prefix(
        pool.ref, _ptr(layer_global_scale), _ptr(block_table), block_table.shape[1],
        _ptr(prefix_lens), _ptr(cu_prefix), prefix_lens.shape[0], int(max_prefix_len),
        _ptr(fp8_scale), _ptr(fp8_k), _ptr(fp8_v), _stream(stream))
    _check(st, "kv4_dequant_prefix")


def kv4_extend_workspace_bytes(batch, max_chunk_len, num_q_heads, head_dim):
    return _load().kv4_extend_workspace_bytes(batch, max_chunk_len, num_q_heads, head_dim)


def alloc_extend_workspace(batch, max_chunk_len, num_q_heads, head_dim, device="cuda"):
    n = kv4_extend_workspace_bytes(batch, max_chunk_len, num_q_heads, head_dim)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device)


def kv4_extend_attention(q, chunk_k, chunk_v, prefix_k, prefix_v, fp8_scale, prefix_lens,
                         cu_prefix, chunk_lens, cu_chunk, max_chunk_len, sm_scale, out,
                         workspace=None, stream=None):
    """Extend attention of the chunk's queries q (bf16 [sum C, Hq, D]) over
    the FP8 prefix workspace plus the FP8 chunk K/V; out is bf16 or float32
    [sum C, Hq, D].  ``workspace`` (alloc_extend_workspace) lets the last
    partial wave of work be split over the SMs."""
    Hq, D = q.shape[1], q.shape[2]
    st = _load().kv4_extend_attention(
        _ptr(q), _ptr(chunk_k), _ptr(chunk_v), _ptr(prefix_k), _ptr(prefix_v), _ptr(fp8_scale),
        _ptr(prefix_lens), _ptr(cu_prefix), _ptr(chunk_lens), _ptr(cu_chunk),
        chunk_lens.shape[0], int(max_chunk_len), Hq, chunk_k.shape[1], D, float(sm_scale),
        _ptr(workspace), workspace.numel() if workspace is not None else 0,
        _ptr(out), 1 if out.dtype == torch.float32 else 0, _stream(stream))
    _check(st, "kv4_extend_attention")


def kv4_k8v4_write(k, v, slot_mapping, pool, key_scale, stream=None):
    """Rotate and quantise bf16 k, v [T, Hkv, D] into a k8v4 ``pool``."""
    st = _load().kv4_k8v4_write(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0], pool.ref,
                                _ptr(key_scale), _stream(stream))
    _check(st, "kv4_k8v4_write")


def kv4_k8v4_workspace_bytes(batch, num_kv_heads, head_dim, num_chunks):
    return _load().kv4_k8v4_workspace_bytes(batch, num_kv_heads, head_dim, num_chunks)


def kv4_k8v4_decode_attention(q, pool, key_scale, block_table, seq_lens, sm_scale, out,
                              num_chunks, workspace, stream=None):
    """Decode attention over a k8v4 pool; ``workspace`` a uint8 CUDA tensor of
    at least kv4_k8v4_workspace_bytes(...) bytes."""
    st = _load().kv4_k8v4_decode_attention(
        _ptr(q), pool.ref, _ptr(key_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        q.shape[0], q.shape[1], float(sm_scale), int(num_chunks), _ptr(workspace),
        workspace.numel() if workspace is not None else 0, _ptr(out),
        1 if out.dtype == torch.float32 else 0, _stream(stream))
    _check(st, "kv4_k8v4_decode_attention")


def kv4_device_error():
    """Read and clear the current device's error word (0 = none)."""
    return _load().kv4_device_error()


def alloc_workspace(batch, num_q_heads, head_dim, num_splits, device="cuda"):
    n = kv4_decode_workspace_bytes(batch, num_q_heads, head_dim, num_splits)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device)
