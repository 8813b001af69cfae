"""Paged KV cache and decode attention for one GB300 GPU (sm_103a).

Thin ctypes binding of libpkv.so (include/pkv.h): it only turns torch
tensors into pointers and sizes and raises on a non-zero status.  Every step
of the path runs in the library's CUDA kernels; there is no fallback.  If
the library is missing it is built in-tree with nvcc, and if that fails the
import of the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "KVError", "KVPool", "BlockAllocator", "PrefixCachePool", "kv_pool_bytes", "slot_mapping", "workspace_bytes",
    "paged_decode_attention", "device_status", "library_path", "load_library", "workspace_init",
    "make_workspace", "paged_decode_append_attention", "paged_prefill_attention", "slot_mapping_varlen",
]

KV_F32, KV_F16, KV_BF16, KV_FP8_E4M3 = 0, 1, 2, 3
DTYPE_CODE = {torch.float32: KV_F32, torch.float16: KV_F16, torch.bfloat16: KV_BF16,
              torch.float8_e4m3fn: KV_FP8_E4M3}
CODE_DTYPE = {v: k for k, v in DTYPE_CODE.items()}
DTYPE_NAMES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
               "e4m3": torch.float8_e4m3fn, "fp8": torch.float8_e4m3fn}
FP8 = torch.float8_e4m3fn
KERNELS = {"auto": 0, "ffma": 1, "mma": 2}
FLAG_BAD_BLOCK_ID, FLAG_BAD_SLOT, FLAG_BAD_CONTEXT, FLAG_TIMEOUT = 0x1, 0x2, 0x4, 0x8

_lock = threading.Lock()
_lib = None


class KVError(RuntimeError):
    """A libpkv call returned a non-zero kv_status_t."""

    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name}: {detail}" if detail else name)
        self.status = status
        self.name = name


class _PoolConfig(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int), ("num_blocks", ctypes.c_int),
                ("block_size", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("device", ctypes.c_int)]


class _DecodeOptions(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("consumer_warps", ctypes.c_int), ("kernel", ctypes.c_int),
                ("heads_per_stage", ctypes.c_int), ("separate_reduce", ctypes.c_int),
                ("no_pdl", ctypes.c_int), ("early_reads", ctypes.c_int), ("test_stall", ctypes.c_int)]


def library_path() -> str:
    return _build.LIBRARY


def _declare(lib):
    P, I, I64, U32P, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                           ctypes.POINTER(ctypes.c_uint32), ctypes.c_size_t)
    sig = {
        "kv_status_string": (ctypes.c_char_p, [I]),
        "kv_last_error": (ctypes.c_char_p, []),
        "kv_pool_bytes": (SZ, [ctypes.POINTER(_PoolConfig)]),
        "kv_pool_create": (I, [ctypes.POINTER(_PoolConfig), P, SZ, ctypes.POINTER(P)]),
        "kv_pool_destroy": (None, [P]),
        "kv_pool_layer": (I, [P, I, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "kv_pool_config": (I, [P, ctypes.POINTER(_PoolConfig)]),
        "kv_slot_mapping": (I, [P, I, P, I, I, I, P, P]),
        "kv_append": (I, [P, I, P, I, P, P, P, P]),
        "paged_decode_workspace_bytes": (I, [I, I, I, I, I, ctypes.POINTER(_DecodeOptions),
                                             ctypes.POINTER(SZ)]),
        "paged_decode_attention": (I, [P, P, P, I, P, I, P, I, I, I, I, I, I, ctypes.c_float, P,
                                       I, P, SZ, ctypes.POINTER(_DecodeOptions), P]),
        "paged_decode_workspace_init": (I, [P, SZ, I, I, P]),
        "paged_decode_append_attention": (I, [P, P, P, P, P, P, I, P, I, P, I, I, I, I, I, I,
                                              ctypes.c_float, P, I, P, P, SZ,
                                              ctypes.POINTER(_DecodeOptions), P]),
        "paged_decode_attention_static": (I, [P, P, P, I, P, I, P, I, I, I, I, I, I, ctypes.c_float,
                                              P, I, ctypes.POINTER(_DecodeOptions), P]),
        "kv_device_status": (I, [I, P, U32P]),
        "kv_allocator_create": (I, [I, I, I, ctypes.POINTER(P)]),
        "kv_allocator_destroy": (None, [P]),
        "kv_allocator_extend": (I, [P, I64, I]),
        "kv_seq_extend": (I, [P, I, I, P, I, ctypes.POINTER(I), P]),
        "kv_seq_free": (I, [P, I]),
        "kv_allocator_release": (I, [P, I64]),
        "kv_allocator_table": (I, [P, I64, ctypes.POINTER(ctypes.c_int32), I,
                                   ctypes.POINTER(I), ctypes.POINTER(I)]),
        "kv_allocator_slot": (I, [P, I64, I, ctypes.POINTER(ctypes.c_int32)]),
        "kv_allocator_free_queue": (I, [P, ctypes.POINTER(ctypes.c_int32), I, ctypes.POINTER(I)]),
        "kv_append_fp8": (I, [P, I, P, I, P, P, I, P, ctypes.c_float, ctypes.c_float, P]),
        "paged_decode_attention_fp8": (I, [P, I, P, P, ctypes.c_float, ctypes.c_float, I, P, I, P, I,
                                           I, I, I, I, ctypes.c_float, P, I, P, SZ,
                                           ctypes.POINTER(_DecodeOptions), P]),
        "paged_decode_append_attention_fp8": (I, [P, P, P, P, I, P, P, ctypes.c_float, ctypes.c_float,
                                                  I, P, I, P, I, I, I, I, I, ctypes.c_float, P, I, P,
                                                  P, SZ, ctypes.POINTER(_DecodeOptions), P]),
        "paged_prefill_workspace_bytes": (SZ, [I]),
        "kv_slot_mapping_varlen": (I, [P, I, P, P, I, I, I, I, P, P]),
        "paged_prefill_attention": (I, [P, P, P, I, P, I, P, P, I, I, I, I, I, I, I, ctypes.c_float, P, I,
                                        P, SZ, P]),
        "paged_prefill_attention_fp8": (I, [P, I, P, P, ctypes.c_float, ctypes.c_float, I, P, I, P, P, I, I, I,
                                            I, I, I, ctypes.c_float, P, I, P, SZ, P]),
        "kv_swap_bytes": (SZ, [P, I]),
        "kv_swap_out": (I, [P, P, I, P, SZ, P]),
        "kv_swap_in": (I, [P, P, I, P, SZ, P]),
        "kv_prefix_pool_create": (I, [I, I, ctypes.POINTER(P)]),
        "kv_prefix_pool_destroy": (None, [P]),
        "kv_prefix_pool_allocate": (I, [P, ctypes.POINTER(ctypes.c_int32), I,
                                        ctypes.POINTER(ctypes.c_int32), I, ctypes.POINTER(I),
                                        ctypes.POINTER(I), ctypes.POINTER(ctypes.c_int32), I,
                                        ctypes.POINTER(I)]),
        "kv_prefix_pool_free": (I, [P, ctypes.POINTER(ctypes.c_int32), I]),
        "kv_prefix_pool_free_queue": (I, [P, ctypes.POINTER(ctypes.c_int32), I, ctypes.POINTER(I)]),
        "kv_prefix_pool_cache_size": (I, [P, ctypes.POINTER(I), ctypes.POINTER(I)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load_library(path: str | None = None):
    """Load libpkv.so (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = _declare(ctypes.CDLL(path or _build.build()))
        if path is None:
            _lib = lib
        return lib


def _check(status: int, lib=None):
    if status != 0:
        lib = lib or load_library()
        raise KVError(status, lib.kv_status_string(status).decode(), lib.kv_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _call_on(t: torch.Tensor, lib, fn, *args):
    """Call a library entry point with t's device current: the library takes
    the SM count, the status word and the static scratch of the current
    device, and the stream passed is t's."""
    if t.device.type != "cuda":  # the library rejects host pointers where it needs device memory
        _check(fn(*args), lib)
        return
    with torch.cuda.device(t.device):
        _check(fn(*args), lib)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def kv_pool_bytes(num_layers, num_blocks, block_size, num_kv_heads, head_dim, dtype) -> int:
    cfg = _PoolConfig(num_layers, num_blocks, block_size, num_kv_heads, head_dim,
                      DTYPE_CODE[dtype], 0)
    return int(load_library().kv_pool_bytes(ctypes.byref(cfg)))


class KVPool:
    """A pool of KV blocks for every layer, in one device buffer owned by torch.

    Layout per layer: K [num_blocks, num_kv_heads, block_size, head_dim], then V.
    """

    def __init__(self, num_layers, num_blocks, block_size, num_kv_heads, head_dim, dtype,
                 device=None, buffer: torch.Tensor | None = None):
        lib = load_library()
        device = torch.device(device if device is not None else "cuda")
        if device.index is None:
            device = torch.device("cuda", torch.cuda.current_device())
        if isinstance(dtype, str):
            _need(dtype in DTYPE_NAMES, f"dtype must be one of {sorted(DTYPE_NAMES)}")
            dtype = DTYPE_NAMES[dtype]
        self.cfg = _PoolConfig(num_layers, num_blocks, block_size, num_kv_heads, head_dim,
                               DTYPE_CODE[dtype], device.index)
        self.nbytes = int(lib.kv_pool_bytes(ctypes.byref(self.cfg)))
        _need(self.nbytes > 0, "invalid pool configuration")
        if buffer is None:
            buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        _need(buffer.dtype == torch.uint8 and buffer.is_contiguous() and buffer.numel() >= self.nbytes,
              "buffer must be a contiguous uint8 tensor of at least kv_pool_bytes bytes")
        self.buffer = buffer
        self.dtype = dtype
        self.device = device
        self.shape = (num_blocks, num_kv_heads, block_size, head_dim)
        handle = ctypes.c_void_p()
        _check(lib.kv_pool_create(ctypes.byref(self.cfg), _ptr(buffer), buffer.numel(),
                                  ctypes.byref(handle)), lib)
        self._handle = handle
        self._lib = lib

    @property
    def num_layers(self):
        return self.cfg.num_layers

    def seq_extend(self, seq_id: int, new_tokens: int, ctx_len: int, max_blocks: int):
        """kv_seq_extend: grow sequence seq_id (currently ctx_len tokens) by
        new_tokens on the pool's own allocator.  Returns (table row [max_blocks]
        padded with -1, new length, slots of the new tokens), host int32 tensors."""
        row = torch.full((max_blocks,), -1, dtype=torch.int32)
        slots = torch.zeros(max(new_tokens, 1), dtype=torch.int32)
        n = ctypes.c_int(ctx_len)
        _check(self._lib.kv_seq_extend(self._handle, seq_id, new_tokens, ctypes.c_void_p(row.data_ptr()),
                                       max_blocks, ctypes.byref(n), ctypes.c_void_p(slots.data_ptr())),
               self._lib)
        return row, n.value, slots[:new_tokens]

    def seq_free(self, seq_id: int):
        """kv_seq_free: return the sequence's blocks to the pool's free queue."""
        _check(self._lib.kv_seq_free(self._handle, seq_id), self._lib)

    def layer(self, layer: int):
        """(K, V) torch views of one layer, addresses taken from kv_pool_layer."""
        k = ctypes.c_void_p()
        v = ctypes.c_void_p()
        _check(self._lib.kv_pool_layer(self._handle, layer, ctypes.byref(k), ctypes.byref(v)),
               self._lib)
        base = self.buffer.data_ptr()
        n = self.nbytes // (2 * self.cfg.num_layers)
        views = []
        for addr in (k.value, v.value):
            off = addr - base
            views.append(self.buffer[off:off + n].view(self.dtype).view(self.shape))
        return views[0], views[1]

    def swap_bytes(self, num_blocks: int) -> int:
        """Bytes of host memory that num_blocks swapped blocks occupy."""
        return int(self._lib.kv_swap_bytes(self._handle, num_blocks))

    def _swap_ids(self, block_ids) -> torch.Tensor:
        if not isinstance(block_ids, torch.Tensor):
            block_ids = torch.tensor(list(block_ids), dtype=torch.int32)
        _need(block_ids.dtype == torch.int32 and block_ids.dim() == 1, "block_ids must be int32 [n]")
        return block_ids.to(self.device).contiguous()

    def swap_out(self, block_ids, host: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Copy the listed blocks (all layers, K and V) into page-locked host memory.

        Returns the host buffer (uint8, kv_swap_bytes(n) bytes; a new pinned
        tensor unless `host` is given).  Asynchronous on `stream`."""
        ids = self._swap_ids(block_ids)
        n = ids.numel()
        need = self.swap_bytes(n)
        if host is None:
            host = torch.empty(max(need, 16), dtype=torch.uint8, pin_memory=True)
        _need(host.dtype == torch.uint8 and host.is_contiguous() and host.numel() >= need,
              "host must be a contiguous uint8 tensor of at least swap_bytes(n) bytes")
        _check(self._lib.kv_swap_out(self._handle, _ptr(ids), n, _ptr(host), host.numel(),
                                     _stream(self.buffer, stream)), self._lib)
        self._swap_keep = ids  # alive until the next swap call on this pool
        return host

    def swap_in(self, block_ids, host: torch.Tensor, stream=None):
        """Copy swapped records from host memory into the listed blocks."""
        ids = self._swap_ids(block_ids)
        n = ids.numel()
        _need(host.dtype == torch.uint8 and host.is_contiguous() and host.numel() >= self.swap_bytes(n),
              "host must be a contiguous uint8 tensor of at least swap_bytes(n) bytes")
        _check(self._lib.kv_swap_in(self._handle, _ptr(ids), n, _ptr(host), host.numel(),
                                    _stream(self.buffer, stream)), self._lib)
        self._swap_keep = ids

    def append(self, layer: int, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
               seq_ids: torch.Tensor | None = None, stream=None, k_scale=None, v_scale=None):
        """Write k, v ([n, Hkv, D]) into this layer at slot_mapping ([n] int32).

        An E4M3 pool quantizes on the way and needs this layer's k_scale and
        v_scale; k and v are then f32, f16 or bf16."""
        n = slot_mapping.shape[0]
        if self.dtype == FP8:
            _need(k_scale is not None and v_scale is not None, "an E4M3 pool needs k_scale and v_scale")
            _need(k.dtype == v.dtype and k.dtype in (torch.float32, torch.float16, torch.bfloat16),
                  "k/v must be f32, f16 or bf16")
            _need(tuple(k.shape) == (n, self.cfg.num_kv_heads, self.cfg.head_dim) and k.shape == v.shape,
                  "k and v must be [n_tokens, num_kv_heads, head_dim]")
            _need(k.is_contiguous() and v.is_contiguous() and slot_mapping.is_contiguous(), "contiguous inputs")
            _need(slot_mapping.dtype == torch.int32, "slot_mapping must be int32")
            _need(seq_ids is None or (seq_ids.dtype == torch.int32 and seq_ids.shape[0] == n),
                  "seq_ids must be int32 [n_tokens]")
            _check(self._lib.kv_append_fp8(self._handle, layer, _ptr(seq_ids), n, _ptr(k), _ptr(v),
                                           DTYPE_CODE[k.dtype], _ptr(slot_mapping), float(k_scale),
                                           float(v_scale), _stream(k, stream)), self._lib)
            return
        _need(k.dtype == self.dtype and v.dtype == self.dtype, "k/v dtype must match the pool")
        _need(tuple(k.shape) == (n, self.cfg.num_kv_heads, self.cfg.head_dim) and k.shape == v.shape,
              "k and v must be [n_tokens, num_kv_heads, head_dim]")
        _need(k.is_contiguous() and v.is_contiguous() and slot_mapping.is_contiguous(), "contiguous inputs")
        _need(slot_mapping.dtype == torch.int32, "slot_mapping must be int32")
        _need(seq_ids is None or (seq_ids.dtype == torch.int32 and seq_ids.shape[0] == n),
              "seq_ids must be int32 [n_tokens]")
        _check(self._lib.kv_append(self._handle, layer, _ptr(seq_ids), n, _ptr(k), _ptr(v),
                                   _ptr(slot_mapping), _stream(k, stream)), self._lib)

    def close(self):
        if getattr(self, "_handle", None):
            self._lib.kv_pool_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def slot_mapping(block_tables: torch.Tensor, context_lens: torch.Tensor, block_size: int,
                 num_blocks: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Device slot of every sequence's newest token (position context_lens - 1)."""
    lib = load_library()
    B = context_lens.shape[0]
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32, "int32 inputs")
    _need(block_tables.is_contiguous() and block_tables.shape[0] == B, "block_tables [B, max_blocks]")
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=context_lens.device)
    _call_on(context_lens, lib, lib.kv_slot_mapping,
             _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B,
             block_size, num_blocks, _ptr(out), _stream(out, stream))
    return out


def _options(num_ctas=0, ctas_per_sm=0, consumer_warps=0, kernel="auto", heads_per_stage=0,
             separate_reduce=False, pdl=True, early_reads=False, test_stall=False) -> _DecodeOptions:
    return _DecodeOptions(num_ctas, ctas_per_sm, consumer_warps, KERNELS[kernel], heads_per_stage,
                          int(separate_reduce), int(not pdl), int(early_reads), int(test_stall))


def workspace_init(workspace: torch.Tensor, num_seqs: int, num_kv_heads: int, stream=None):
    """Zero the merge counters at the start of a workspace (once after allocation)."""
    lib = load_library()
    _call_on(workspace, lib, lib.paged_decode_workspace_init,
             _ptr(workspace), workspace.numel(), num_seqs, num_kv_heads,
                                           _stream(workspace, stream))


def make_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, device=None, **opts) -> torch.Tensor:
    """A zero-filled workspace for paged_decode_attention with these sizes and options."""
    dev = torch.device(device if device is not None else "cuda")
    n = workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, dev, **opts)
    return torch.zeros(n, dtype=torch.uint8, device=dev)


def workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, device=None, **opts) -> int:
    lib = load_library()
    dev = torch.device(device if device is not None else "cuda")
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    o = _options(**opts)
    n = ctypes.c_size_t()
    _check(lib.paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, idx,
                                            ctypes.byref(o), ctypes.byref(n)), lib)
    return int(n.value)


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           out=None, out_dtype=None, workspace=None, stream=None, k_scale=None,
                           v_scale=None, **opts):
    """out[s, g] = softmax(scale q[s, g] . K_s^T) V_s over the paged cache (one layer).

    q [B, Hq, D]; k_cache/v_cache [NB, Hkv, bs, D]; block_tables int32 [B, max_blocks];
    context_lens int32 [B].  opts: num_ctas, ctas_per_sm, consumer_warps, kernel.
    E4M3 (torch.float8_e4m3fn) caches stand for k_scale (v_scale) times their codes.
    """
    lib = load_library()
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    _need(D == D2 and tuple(v_cache.shape) == tuple(k_cache.shape), "cache shapes")
    fp8 = k_cache.dtype == FP8
    if fp8:
        _need(v_cache.dtype == FP8 and k_scale is not None and v_scale is not None,
              "an E4M3 cache needs both caches E4M3 and k_scale, v_scale")
    else:
        _need(q.dtype == k_cache.dtype == v_cache.dtype, "q and the caches share a dtype")
    _need(all(t.is_contiguous() for t in (q, k_cache, v_cache, block_tables, context_lens)),
          "contiguous inputs")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32, "int32 tables")
    _need(block_tables.shape[0] == B and context_lens.shape[0] == B, "one table row and length per sequence")
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    _need(out.dtype == out_dtype and tuple(out.shape) == (B, Hq, D) and out.is_contiguous(), "out")
    o = _options(**opts)
    if workspace is None:
        workspace = make_workspace(B, Hq, Hkv, D, q.device, **opts)
    if fp8:
        _call_on(q, lib, lib.paged_decode_attention_fp8,
            _ptr(q), DTYPE_CODE[q.dtype], _ptr(k_cache), _ptr(v_cache), float(k_scale), float(v_scale),
            NB, _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs,
            float(scale), _ptr(out), DTYPE_CODE[out_dtype], _ptr(workspace), workspace.numel(),
            ctypes.byref(o), _stream(q, stream))
        return out
    _call_on(q, lib, lib.paged_decode_attention,
        _ptr(q), _ptr(k_cache), _ptr(v_cache), NB, _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, Hq, Hkv, D, bs, DTYPE_CODE[q.dtype], float(scale), _ptr(out),
        DTYPE_CODE[out_dtype], _ptr(workspace), workspace.numel(), ctypes.byref(o),
        _stream(q, stream))
    return out


def paged_decode_append_attention(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                                  scale: float, seq_ids=None, out=None, out_dtype=None,
                                  slot_mapping=None, workspace=None, stream=None, k_scale=None,
                                  v_scale=None, **opts):
    """One layer of a decode step in one kernel: append k_new/v_new ([B, Hkv, D]) at
    position context_lens - 1 of every sequence, then attend (see paged_decode_attention).

    seq_ids: optional int32 [B]; a negative entry skips the append of that sequence.
    slot_mapping: optional int32 [B] output receiving the newest-token slots.
    """
    lib = load_library()
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    _need(D == D2 and tuple(v_cache.shape) == tuple(k_cache.shape), "cache shapes")
    fp8 = k_cache.dtype == FP8
    if fp8:
        _need(v_cache.dtype == FP8 and k_scale is not None and v_scale is not None,
              "an E4M3 cache needs both caches E4M3 and k_scale, v_scale")
        _need(q.dtype == k_new.dtype == v_new.dtype, "q, k_new and v_new share a dtype")
    else:
        _need(q.dtype == k_cache.dtype == v_cache.dtype == k_new.dtype == v_new.dtype, "one dtype")
    _need(tuple(k_new.shape) == (B, Hkv, D) and k_new.shape == v_new.shape, "k_new/v_new [B, Hkv, D]")
    _need(all(t.is_contiguous() for t in (q, k_new, v_new, k_cache, v_cache, block_tables, context_lens)),
          "contiguous inputs")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32, "int32 tables")
    _need(block_tables.shape[0] == B and context_lens.shape[0] == B, "one table row and length per sequence")
    _need(seq_ids is None or (seq_ids.dtype == torch.int32 and seq_ids.shape[0] == B), "seq_ids int32 [B]")
    _need(slot_mapping is None or (slot_mapping.dtype == torch.int32 and slot_mapping.shape[0] == B),
          "slot_mapping int32 [B]")
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    _need(out.dtype == out_dtype and tuple(out.shape) == (B, Hq, D) and out.is_contiguous(), "out")
    o = _options(**opts)
    if workspace is None:
        workspace = make_workspace(B, Hq, Hkv, D, q.device, **opts)
    if fp8:
        _call_on(q, lib, lib.paged_decode_append_attention_fp8,
            _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(seq_ids), DTYPE_CODE[q.dtype], _ptr(k_cache),
            _ptr(v_cache), float(k_scale), float(v_scale), NB, _ptr(block_tables), block_tables.shape[1],
            _ptr(context_lens), B, Hq, Hkv, D, bs, float(scale), _ptr(out), DTYPE_CODE[out_dtype],
            _ptr(slot_mapping), _ptr(workspace), workspace.numel(), ctypes.byref(o),
            _stream(q, stream))
        return out
    _call_on(q, lib, lib.paged_decode_append_attention,
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(seq_ids), _ptr(k_cache), _ptr(v_cache), NB,
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs,
        DTYPE_CODE[q.dtype], float(scale), _ptr(out), DTYPE_CODE[out_dtype], _ptr(slot_mapping),
        _ptr(workspace), workspace.numel(), ctypes.byref(o), _stream(q, stream))
    return out


def slot_mapping_varlen(block_tables: torch.Tensor, query_start: torch.Tensor, context_lens: torch.Tensor,
                        block_size: int, num_blocks: int, num_tokens: int | None = None,
                        out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Device slot of every new token of a multi-token step (int32 [num_tokens])."""
    lib = load_library()
    B = context_lens.shape[0]
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32 and
          query_start.dtype == torch.int32, "int32 inputs")
    _need(query_start.shape[0] == B + 1 and block_tables.shape[0] == B and block_tables.is_contiguous(),
          "query_start [B + 1], block_tables [B, max_blocks]")
    if num_tokens is None:
        num_tokens = int(query_start[-1].item())
    if out is None:
        out = torch.empty(max(num_tokens, 1), dtype=torch.int32, device=context_lens.device)[:num_tokens]
    _call_on(context_lens, lib, lib.kv_slot_mapping_varlen,
             _ptr(block_tables), block_tables.shape[1], _ptr(query_start),
             _ptr(context_lens), B, num_tokens, block_size, num_blocks, _ptr(out),
             _stream(context_lens, stream))
    return out


def paged_prefill_attention(q, k_cache, v_cache, block_tables, query_start, context_lens, scale: float,
                            out=None, out_dtype=None, workspace=None, stream=None, k_scale=None, v_scale=None):
    """Causal attention of a step's new tokens (q [T, Hq, D], rows grouped by
    sequence as query_start says) over the paged cache they were appended to.
    E4M3 (torch.float8_e4m3fn) caches stand for k_scale (v_scale) times their codes."""
    lib = load_library()
    T, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    B = context_lens.shape[0]
    _need(D == D2 and tuple(v_cache.shape) == tuple(k_cache.shape), "cache shapes")
    fp8 = k_cache.dtype == FP8
    if fp8:
        _need(v_cache.dtype == FP8 and k_scale is not None and v_scale is not None,
              "an E4M3 cache needs both caches E4M3 and k_scale, v_scale")
    else:
        _need(q.dtype == k_cache.dtype == v_cache.dtype, "q and the caches share a dtype")
    _need(all(t.is_contiguous() for t in (q, k_cache, v_cache, block_tables, query_start, context_lens)),
          "contiguous inputs")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32 and
          query_start.dtype == torch.int32, "int32 tables")
    _need(block_tables.shape[0] == B and query_start.shape[0] == B + 1, "table rows / query_start")
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((T, Hq, D), dtype=out_dtype, device=q.device)
    _need(out.dtype == out_dtype and tuple(out.shape) == (T, Hq, D) and out.is_contiguous(), "out")
    if workspace is None:
        workspace = torch.empty(max(16, int(lib.paged_prefill_workspace_bytes(B))), dtype=torch.uint8,
                                device=q.device)
    if fp8:
        _call_on(q, lib, lib.paged_prefill_attention_fp8,
                 _ptr(q), DTYPE_CODE[q.dtype], _ptr(k_cache), _ptr(v_cache), float(k_scale), float(v_scale), NB,
                 _ptr(block_tables), block_tables.shape[1], _ptr(query_start), _ptr(context_lens), B, T, Hq, Hkv,
                 D, bs, float(scale), _ptr(out), DTYPE_CODE[out_dtype], _ptr(workspace), workspace.numel(),
                 _stream(q, stream))
        return out
    _call_on(q, lib, lib.paged_prefill_attention,
        _ptr(q), _ptr(k_cache), _ptr(v_cache), NB, _ptr(block_tables), block_tables.shape[1],
        _ptr(query_start), _ptr(context_lens), B, T, Hq, Hkv, D, bs, DTYPE_CODE[q.dtype], float(scale),
        _ptr(out), DTYPE_CODE[out_dtype], _ptr(workspace), workspace.numel(), _stream(q, stream))
    return out


def paged_decode_attention_static(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                                  out=None, out_dtype=None, stream=None, **opts):
    """paged_decode_attention with the library's fixed device scratch instead of a
    workspace: the call allocates nothing (see include/pkv.h)."""
    lib = load_library()
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    _need(D == D2 and tuple(v_cache.shape) == tuple(k_cache.shape), "cache shapes")
    _need(q.dtype == k_cache.dtype == v_cache.dtype, "q and the caches share a dtype")
    _need(all(t.is_contiguous() for t in (q, k_cache, v_cache, block_tables, context_lens)),
          "contiguous inputs")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32, "int32 tables")
    out_dtype = out_dtype or q.dtype
    _need(out is not None, "out must be given (the call allocates nothing)")
    _need(out.dtype == out_dtype and tuple(out.shape) == (B, Hq, D) and out.is_contiguous(), "out")
    o = _options(**opts)
    _call_on(q, lib, lib.paged_decode_attention_static,
        _ptr(q), _ptr(k_cache), _ptr(v_cache), NB, _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, Hq, Hkv, D, bs, DTYPE_CODE[q.dtype], float(scale), _ptr(out),
        DTYPE_CODE[out_dtype], ctypes.byref(o), _stream(q, stream))
    return out


def device_status(device=None, stream=None):
    """Synchronise, then read and clear the device status word: (status, flags)."""
    lib = load_library()
    dev = torch.device(device if device is not None else "cuda")
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    s = stream if stream is not None else torch.cuda.current_stream(idx)
    flags = ctypes.c_uint32()
    st = lib.kv_device_status(idx, ctypes.c_void_p(s.cuda_stream), ctypes.byref(flags))
    return int(st), int(flags.value)


class BlockAllocator:
    """Host block allocator (FIFO free queue, optional null block 0)."""

    def __init__(self, num_blocks: int, block_size: int, reserve_null_block: bool = True):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check(self._lib.kv_allocator_create(num_blocks, block_size, int(reserve_null_block),
                                             ctypes.byref(h)), self._lib)
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def extend(self, seq_id: int, new_tokens: int) -> bool:
        """Room for new_tokens more tokens; False (nothing changed) when blocks run out."""
        st = self._lib.kv_allocator_extend(self._h, seq_id, new_tokens)
        if st == 4:  # KV_ERR_OUT_OF_BLOCKS
            return False
        _check(st, self._lib)
        return True

    def release(self, seq_id: int):
        _check(self._lib.kv_allocator_release(self._h, seq_id), self._lib)

    def table(self, seq_id: int):
        nb, nt = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.kv_allocator_table(self._h, seq_id, None, 0, ctypes.byref(nb),
                                            ctypes.byref(nt)), self._lib)
        buf = (ctypes.c_int32 * max(1, nb.value))()
        _check(self._lib.kv_allocator_table(self._h, seq_id, buf, nb.value, None, None), self._lib)
        return list(buf[:nb.value]), nt.value

    def slot(self, seq_id: int, position: int) -> int:
        out = ctypes.c_int32()
        _check(self._lib.kv_allocator_slot(self._h, seq_id, position, ctypes.byref(out)), self._lib)
        return int(out.value)

    def free_queue(self):
        n = ctypes.c_int()
        _check(self._lib.kv_allocator_free_queue(self._h, None, 0, ctypes.byref(n)), self._lib)
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check(self._lib.kv_allocator_free_queue(self._h, buf, n.value, None), self._lib)
        return list(buf[:n.value])

    def __del__(self):
        try:
            if getattr(self, "_h", None):
                self._lib.kv_allocator_destroy(self._h)
                self._h = None
        except Exception:
            pass


class PrefixCachePool:
    """Host block pool with prefix caching (chained block hashes, LRU free queue)."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check(self._lib.kv_prefix_pool_create(num_blocks, block_size, ctypes.byref(h)), self._lib)
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def allocate(self, tokens):
        """Blocks for a request with these token ids: (blocks, cached_tokens, evicted).

        Returns None (nothing changed) when too few blocks are free."""
        tokens = [int(t) for t in tokens]
        n = len(tokens)
        cap = max(1, -(-n // self.block_size))
        tok = (ctypes.c_int32 * max(1, n))(*tokens)
        blocks = (ctypes.c_int32 * cap)()
        evicted = (ctypes.c_int32 * cap)()
        nb, cached, ne = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        st = self._lib.kv_prefix_pool_allocate(self._h, tok, n, blocks, cap, ctypes.byref(nb),
                                               ctypes.byref(cached), evicted, cap, ctypes.byref(ne))
        if st == 4:  # KV_ERR_OUT_OF_BLOCKS
            return None
        _check(st, self._lib)
        return list(blocks[:nb.value]), int(cached.value), list(evicted[:ne.value])

    def free(self, blocks):
        blocks = [int(b) for b in blocks]
        buf = (ctypes.c_int32 * max(1, len(blocks)))(*blocks)
        _check(self._lib.kv_prefix_pool_free(self._h, buf, len(blocks)), self._lib)

    def free_queue(self):
        n = ctypes.c_int()
        _check(self._lib.kv_prefix_pool_free_queue(self._h, None, 0, ctypes.byref(n)), self._lib)
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check(self._lib.kv_prefix_pool_free_queue(self._h, buf, n.value, None), self._lib)
        return list(buf[:n.value])

    def cache_size(self):
        h, b = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.kv_prefix_pool_cache_size(self._h, ctypes.byref(h), ctypes.byref(b)),
               self._lib)
        return int(h.value), int(b.value)

    def __del__(self):
        try:
            if getattr(self, "_h", None):
                self._lib.kv_prefix_pool_destroy(self._h)
                self._h = None
        except Exception:
            pass
