"""Oracle for one paged-KV decode step: plain C, fp64 (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  The CUDA library never imports, links or calls it, and it
never calls the CUDA library: the two share only the seeded inputs of
`workloads`.

Functions and the passage each follows (see pkv_oracle.c for the C side):
  slot_mapping  -- "vLLM Architecture and Installation", Example 3
  append        -- same Example 3 (new K/V go to the slot of each token)
  paged_decode  -- same Example 3 (history read through the block table) and
                   "Batching and Scheduling", Example 1 (each sequence reads its
                   own KV every step); softmax(scale q.K^T).V in fp64.
  paged_prefill, slot_mapping_varlen
                -- multi-token queries (chunked prefill: "Batching and
                   Scheduling", Example 5; "vLLM Architecture and Installation",
                   Example 5): new token i of a sequence with context c and n
                   new tokens sits at position c - n + i and attends causally
                   to positions 0 .. c - n + i.
  e4m3_encode, quantize_e4m3, append_e4m3, paged_decode(k_scale, v_scale)
                -- the FP8 KV cache of "vLLM Architecture and Installation",
                   Example 6 (one byte per value): E4M3 codes with one fp32
                   scale per layer for K and for V (the pages fix the byte
                   count, not the format; see pkv_oracle.c).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pkv_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")
DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}
_lock = threading.Lock()
_lib = None


def build(source: str = SOURCE, output: str = LIBRARY, extra_flags=(), force=False) -> str:
    """Compile the oracle with gcc into a shared library (no CUDA involved)."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-D_POSIX_C_SOURCE=200809L", *extra_flags, source, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


def load(path: str | None = None):
    """Load (building first if needed) and declare the C entry points."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(build() if path is None else path)
        c_p, c_i, c_i64, c_d = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_decode.argtypes = [c_i, c_p, c_i64, c_p]
        lib.oracle_decode.restype = None
        lib.oracle_slot.argtypes = [c_p, c_i, c_i, c_i, c_i]
        lib.oracle_slot.restype = c_i64
        lib.oracle_slot_mapping.argtypes = [c_p, c_i, c_p, c_i, c_i, c_p]
        lib.oracle_slot_mapping.restype = None
        lib.oracle_append.argtypes = [c_i, c_i, c_i, c_i, c_i, c_p, c_p, c_i, c_p, c_p, c_p]
        lib.oracle_append.restype = c_i
        lib.oracle_paged_decode.argtypes = [c_i, c_p, c_p, c_p, c_p, c_i, c_p, c_i, c_i, c_i,
                                            c_i, c_i, c_i, c_d, c_p, c_i]
        lib.oracle_paged_decode.restype = c_i
        lib.oracle_paged_decode_scaled.argtypes = [c_i, c_i, c_d, c_d, c_p, c_p, c_p, c_p, c_i, c_p,
                                                   c_i, c_i, c_i, c_i, c_i, c_i, c_d, c_p, c_i]
        lib.oracle_paged_decode_scaled.restype = c_i
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize_e4m3.argtypes = [c_i, c_p, c_i64, ctypes.c_float, c_p]
        lib.oracle_quantize_e4m3.restype = None
        lib.oracle_append_e4m3.argtypes = [c_i, c_i, c_i, c_i, c_i, c_p, c_p, c_i, c_p, c_p, c_p,
                                           ctypes.c_float, ctypes.c_float]
        lib.oracle_append_e4m3.restype = c_i
        lib.oracle_paged_prefill.argtypes = [c_i, c_p, c_p, c_p, c_p, c_i, c_p, c_p, c_i, c_i, c_i, c_i,
                                             c_i, c_i, c_d, c_p, c_i]
        lib.oracle_paged_prefill.restype = c_i
        lib.oracle_paged_prefill_scaled.argtypes = [c_i, c_i, c_d, c_d, c_p, c_p, c_p, c_p, c_i, c_p, c_p, c_i,
                                                    c_i, c_i, c_i, c_i, c_i, c_d, c_p, c_i]
        lib.oracle_paged_prefill_scaled.restype = c_i
        lib.oracle_slot_mapping_varlen.argtypes = [c_p, c_i, c_p, c_p, c_i, c_i, c_p]
        lib.oracle_slot_mapping_varlen.restype = None
        lib.oracle_num_cores.argtypes = []
        lib.oracle_num_cores.restype = c_i
        if path is None:
            _lib = lib
        return lib


def _raw(t) -> np.ndarray:
    """Contiguous host bytes of a tensor/array (bf16 kept as its bit pattern)."""
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy()
        if t.dtype == torch.float8_e4m3fn:
            return t.view(torch.uint8).numpy()
        return t.numpy()
    return np.ascontiguousarray(t)


def _dtype_name(t) -> str:
    if isinstance(t, torch.Tensor):
        return {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16",
                torch.float8_e4m3fn: "e4m3"}[t.dtype]
    return {np.dtype(np.float32): "f32", np.dtype(np.float16): "f16"}[np.asarray(t).dtype]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def decode_values(bits, dtype: str, lib=None) -> np.ndarray:
    lib = lib or load()
    a = np.ascontiguousarray(bits)
    out = np.empty(a.size, dtype=np.float64)
    lib.oracle_decode(DTYPE_CODE[dtype], _ptr(a), a.size, _ptr(out))
    return out.reshape(a.shape)


def slot(block_tables, seq: int, position: int, block_size: int, lib=None) -> int:
    lib = lib or load()
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    return int(lib.oracle_slot(_ptr(t), t.shape[1], seq, position, block_size))


def slot_mapping(block_tables, context_lens, block_size: int, lib=None) -> np.ndarray:
    lib = lib or load()
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    c = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty(len(c), dtype=np.int32)
    lib.oracle_slot_mapping(_ptr(t), t.shape[1], _ptr(c), len(c), block_size, _ptr(out))
    return out


def append(k_cache, v_cache, k_new, v_new, slots, lib=None):
    """Scatter k_new/v_new ([n, Hkv, D]) into copies of the pools; returns (K, V) as torch tensors."""
    lib = lib or load()
    dt = _dtype_name(k_cache)
    kc = _raw(k_cache).copy()
    vc = _raw(v_cache).copy()
    kn, vn = _raw(k_new), _raw(v_new)
    sl = np.ascontiguousarray(slots, dtype=np.int32)
    NB, Hkv, bs, D = kc.shape
    rc = lib.oracle_append(DTYPE_CODE[dt], NB, bs, Hkv, D, _ptr(kc), _ptr(vc), len(sl),
                           _ptr(kn), _ptr(vn), _ptr(sl))
    if rc != 0:
        raise ValueError("oracle_append: slot outside the pool")
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]
    if dt == "bf16":
        return (torch.from_numpy(kc).view(torch.bfloat16), torch.from_numpy(vc).view(torch.bfloat16))
    return torch.from_numpy(kc).to(tdt), torch.from_numpy(vc).to(tdt)


def e4m3_encode(x: float, lib=None) -> int:
    """Nearest E4M3 code of the binary32 value x (ties to even, saturating)."""
    return int((lib or load()).oracle_e4m3_encode(float(x)))


def quantize_e4m3(x, scale: float, lib=None) -> torch.Tensor:
    """E4M3 codes of x / scale (fp32 quotient), as a float8_e4m3fn tensor of x's shape."""
    lib = lib or load()
    a = _raw(x)
    out = np.empty(a.size, dtype=np.uint8)
    lib.oracle_quantize_e4m3(DTYPE_CODE[_dtype_name(x)], _ptr(a), a.size, float(scale), _ptr(out))
    return torch.from_numpy(out.reshape(a.shape)).view(torch.float8_e4m3fn)


def append_e4m3(k_cache, v_cache, k_new, v_new, slots, k_scale: float, v_scale: float, lib=None):
    """Quantize k_new/v_new ([n, Hkv, D]) into copies of E4M3 pools; returns (K, V)."""
    lib = lib or load()
    if _dtype_name(k_cache) != "e4m3":
        raise ValueError("append_e4m3 needs float8_e4m3fn pools")
    kc = _raw(k_cache).copy()
    vc = _raw(v_cache).copy()
    kn, vn = _raw(k_new), _raw(v_new)
    sl = np.ascontiguousarray(slots, dtype=np.int32)
    NB, Hkv, bs, D = kc.shape
    rc = lib.oracle_append_e4m3(DTYPE_CODE[_dtype_name(k_new)], NB, bs, Hkv, D, _ptr(kc), _ptr(vc),
                                len(sl), _ptr(kn), _ptr(vn), _ptr(sl), float(k_scale), float(v_scale))
    if rc != 0:
        raise ValueError("oracle_append_e4m3: slot outside the pool")
    return (torch.from_numpy(kc).view(torch.float8_e4m3fn), torch.from_numpy(vc).view(torch.float8_e4m3fn))


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 nthreads: int = 0, lib=None, k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """fp64 output [B, Hq, D] of single-query attention over the paged cache.

    An E4M3 cache stands for k_scale (v_scale) times its codes' values; other
    caches share q's dtype and take no scales."""
    lib = lib or load()
    dt = _dtype_name(k_cache)
    qdt = _dtype_name(q)
    if dt == "e4m3":
        qa, kc, vc = _raw(q), _raw(k_cache), _raw(v_cache)
        t = np.ascontiguousarray(block_tables, dtype=np.int32)
        c = np.ascontiguousarray(context_lens, dtype=np.int32)
        B, Hq, D = qa.shape
        NB, Hkv, bs, D2 = kc.shape
        assert D == D2 and t.shape[0] == B and len(c) == B
        out = np.empty((B, Hq, D), dtype=np.float64)
        rc = lib.oracle_paged_decode_scaled(DTYPE_CODE[qdt], DTYPE_CODE[dt], float(k_scale),
                                            float(v_scale), _ptr(qa), _ptr(kc), _ptr(vc), _ptr(t),
                                            t.shape[1], _ptr(c), B, Hq, Hkv, D, bs, NB, float(scale),
                                            _ptr(out), nthreads)
        if rc != 0:
            raise ValueError(f"oracle_paged_decode_scaled failed ({rc})")
        return out
    if qdt != dt or k_scale != 1.0 or v_scale != 1.0:
        raise ValueError("q and a non-E4M3 cache must share a dtype and take no scales")
    qa, kc, vc = _raw(q), _raw(k_cache), _raw(v_cache)
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    c = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = qa.shape
    NB, Hkv, bs, D2 = kc.shape
    assert D == D2 and t.shape[0] == B and len(c) == B
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = lib.oracle_paged_decode(DTYPE_CODE[dt], _ptr(qa), _ptr(kc), _ptr(vc), _ptr(t), t.shape[1],
                                 _ptr(c), B, Hq, Hkv, D, bs, NB, float(scale), _ptr(out), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_paged_decode failed ({rc})")
    return out


def slot_mapping_varlen(block_tables, query_start, context_lens, block_size: int, lib=None) -> np.ndarray:
    """Slot of every new token of a multi-token step ([T] int32)."""
    lib = lib or load()
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    c = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty(int(qs[-1]), dtype=np.int32)
    lib.oracle_slot_mapping_varlen(_ptr(t), t.shape[1], _ptr(qs), _ptr(c), len(c), block_size, _ptr(out))
    return out


def paged_prefill(q, k_cache, v_cache, block_tables, query_start, context_lens, scale: float,
                  nthreads: int = 0, lib=None, k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """fp64 output [T, Hq, D] of multi-token (causal) queries over the paged cache.

    An E4M3 cache stands for k_scale (v_scale) times its codes' values; other
    caches share q's dtype and take no scales."""
    lib = lib or load()
    dt = _dtype_name(k_cache)
    qdt = _dtype_name(q)
    if dt != "e4m3" and (qdt != dt or k_scale != 1.0 or v_scale != 1.0):
        raise ValueError("q and a non-E4M3 cache must share a dtype and take no scales")
    qa, kc, vc = _raw(q), _raw(k_cache), _raw(v_cache)
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    c = np.ascontiguousarray(context_lens, dtype=np.int32)
    T, Hq, D = qa.shape
    NB, Hkv, bs, D2 = kc.shape
    B = len(c)
    assert D == D2 and t.shape[0] == B and len(qs) == B + 1 and int(qs[-1]) == T
    out = np.empty((T, Hq, D), dtype=np.float64)
    rc = lib.oracle_paged_prefill_scaled(DTYPE_CODE[qdt], DTYPE_CODE[dt], float(k_scale), float(v_scale),
                                         _ptr(qa), _ptr(kc), _ptr(vc), _ptr(t), t.shape[1], _ptr(qs), _ptr(c), B,
                                         Hq, Hkv, D, bs, NB, float(scale), _ptr(out), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_paged_prefill_scaled failed ({rc})")
    return out


def num_cores(lib=None) -> int:
    return int((lib or load()).oracle_num_cores())
