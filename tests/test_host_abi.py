"""CPU-only tests of the C ABI: symbols, sizes, validation, host allocator.

No test here launches anything on a GPU: every call either stays on the host
(sizes, allocator, pool bookkeeping over an adopted fake address) or fails in
argument validation, which runs before any CUDA call.
"""
import ctypes
import json
import os
import re

import pytest
import torch

import paged_kv_cache_slots_gb300 as pkv
from paged_kv_cache_slots_gb300 import roofline

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def declared_functions():
    with open(os.path.join(ROOT, "include", "pkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:kv|paged)_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return pkv.load_library()


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 19
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in range(10):
        assert lib.kv_status_string(code).decode().startswith("KV_")
    assert lib.kv_status_string(0) == b"KV_OK"


@pytest.mark.parametrize("case", _golden("kv_sizes.json")["cases"], ids=lambda c: c["what"][:40])
def test_pool_bytes_match_the_pages(case):
    if case["elem_bytes"] == 1:
        # FP8 pools are not a dtype of this library; the formula is checked
        # through the byte model instead.
        per = roofline.kv_bytes_per_token(case["num_layers"], case["num_kv_heads"], case["head_dim"], 1)
        assert per * case["num_blocks"] * case["block_size"] == case["bytes"]
        return
    dtype = torch.float16
    got = pkv.kv_pool_bytes(case["num_layers"], case["num_blocks"], case["block_size"],
                            case["num_kv_heads"], case["head_dim"], dtype)
    assert got == case["bytes"]
    per = roofline.kv_bytes_per_token(case["num_layers"], case["num_kv_heads"], case["head_dim"],
                                      case["elem_bytes"])
    assert per * case["num_blocks"] * case["block_size"] == case["bytes"]


def test_decode_roofline_reproduces_the_printed_table():
    g = _golden("decode_roofline_rtx4090.json")
    for row in g["rows"]:
        r = roofline.decode_step_roofline(row["batch"], g["params"], g["bits_per_weight"], g["context"],
                                          g["kv_bytes_per_token"], g["peak_flops"], g["bandwidth"])
        assert f"{r['bytes'] / 1e9:.2f}" == f"{row['bytes_gb']:.2f}"
        assert f"{r['step_s'] * 1e3:.2f}" == f"{row['step_ms']:.2f}"
        assert f"{r['tok_s']:.0f}" == f"{row['tok_s']:.0f}"
        assert f"{r['tok_s_per_seq']:.1f}" == f"{row['tok_s_per_seq']:.1f}"
        assert f"{100 * r['util']:.2f}" == f"{row['util_pct']:.2f}"
    r32 = roofline.decode_step_roofline(32, g["params"], g["bits_per_weight"], g["context"],
                                        g["kv_bytes_per_token"], g["peak_flops"], g["bandwidth"])
    assert f"{r32['kv_bytes'] / 1e9:.2f}" == f"{g['kv_gb_at_batch_32']:.2f}"
    assert roofline.sequences_that_fit(g["vram"], g["params"], g["bits_per_weight"], g["context"],
                                       g["kv_bytes_per_token"]) == g["fit_sequences"]


def test_attention_bytes_of_the_batch32_step():
    # 32 layers x 32 sequences x 4096 tokens x 128 KiB/token / 32 layers per layer.
    b = roofline.attention_bytes([4096] * 32, 32, 8, 128, 2, 16, 2, appended_tokens=32)
    assert b.kv * 32 == 32 * 4096 * 131072
    assert b.tables == 32 * 256 * 4


def test_block_allocator_reproduces_the_worked_example():
    g = _golden("block_tables_vllm_example3.json")
    a = pkv.BlockAllocator(g["num_blocks"], g["block_size"], g["reserve_null_block"])
    ids = {}

    def sid(name):
        return ids.setdefault(name, len(ids) + 100)

    for step in g["steps"]:
        op = step["op"]
        if op == "extend":
            assert a.extend(sid(step["seq"]), step["tokens"]) == step["ok"], step
        elif op == "free":
            a.release(sid(step["seq"]))
        elif op == "check":
            assert a.free_queue() == step["free"], step["label"]
            for name, table in step["tables"].items():
                t, n = a.table(sid(name))
                assert t == table and n == step["lengths"][name], (step["label"], name)
            live = set(step["tables"])
            for name in ids:
                if name not in live:
                    with pytest.raises(pkv.KVError):
                        a.table(sid(name))
        elif op == "slots":
            for name, pos, slot in step["expect"]:
                assert a.slot(sid(name), pos) == slot
        elif op == "unused_slots":
            waste = 0
            for name in ("A", "B"):
                t, n = a.table(sid(name))
                waste += len(t) * g["block_size"] - n
            assert waste == step["expect"]


def test_allocator_exhaustion_and_errors():
    a = pkv.BlockAllocator(4, 16, reserve_null_block=False)
    assert a.extend(1, 64)  # all four blocks
    assert not a.extend(2, 1)  # nothing left, nothing changes
    with pytest.raises(pkv.KVError):
        a.table(2)
    assert a.free_queue() == []
    a.release(1)
    assert a.free_queue() == [0, 1, 2, 3]
    with pytest.raises(pkv.KVError) as e:
        a.release(1)
    assert e.value.name == "KV_ERR_NOT_FOUND"
    with pytest.raises(pkv.KVError):
        a.slot(7, 0)


def _cfg(**kw):
    base = dict(num_layers=3, num_blocks=10, block_size=16, num_kv_heads=2, head_dim=64, dtype=1, device=0)
    base.update(kw)
    return pkv._PoolConfig(**base)


def test_pool_adopts_a_buffer_and_lays_out_layers(lib):
    cfg = _cfg()
    n = lib.kv_pool_bytes(ctypes.byref(cfg))
    assert n == 2 * 3 * 10 * 16 * 2 * 64 * 2
    fake = 0x10000000  # adopted, never dereferenced on the host
    h = ctypes.c_void_p()
    assert lib.kv_pool_create(ctypes.byref(cfg), ctypes.c_void_p(fake), n, ctypes.byref(h)) == 0
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    per = n // 6
    for layer in range(3):
        assert lib.kv_pool_layer(h, layer, ctypes.byref(k), ctypes.byref(v)) == 0
        assert k.value == fake + 2 * layer * per and v.value == fake + (2 * layer + 1) * per
    assert lib.kv_pool_layer(h, 3, ctypes.byref(k), ctypes.byref(v)) == 1
    lib.kv_pool_destroy(h)
    # Too small, misaligned, bad shapes.
    assert lib.kv_pool_create(ctypes.byref(cfg), ctypes.c_void_p(fake), n - 1, ctypes.byref(h)) == 1
    assert lib.kv_pool_create(ctypes.byref(cfg), ctypes.c_void_p(fake + 8), n, ctypes.byref(h)) == 1
    assert lib.kv_pool_create(ctypes.byref(_cfg(head_dim=4)), ctypes.c_void_p(fake), n, ctypes.byref(h)) == 1
    assert lib.kv_pool_bytes(ctypes.byref(_cfg(dtype=7))) == 0


def test_pool_sequence_bookkeeping(lib):
    # kv_seq_extend / kv_seq_free on the pool's own allocator: blocks taken from
    # the front of the free queue only when a token crosses a block boundary,
    # slots = block * block_size + offset, tables padded with -1, released
    # blocks to the back of the queue ("vLLM Architecture and Installation",
    # Example 3).  The pool adopts a fake device address (never dereferenced).
    cfg = _cfg()  # 10 blocks of 16 tokens
    n = lib.kv_pool_bytes(ctypes.byref(cfg))
    h = ctypes.c_void_p()
    assert lib.kv_pool_create(ctypes.byref(cfg), ctypes.c_void_p(0x10000000), n, ctypes.byref(h)) == 0
    row = (ctypes.c_int32 * 4)()
    slots = (ctypes.c_int32 * 40)()
    ln = ctypes.c_int(0)
    assert lib.kv_seq_extend(h, 7, 20, row, 4, ctypes.byref(ln), slots) == 0
    assert ln.value == 20 and list(row) == [0, 1, -1, -1]
    assert list(slots[:20]) == list(range(20))
    ln2 = ctypes.c_int(0)
    assert lib.kv_seq_extend(h, 3, 5, row, 4, ctypes.byref(ln2), slots) == 0
    assert list(row) == [2, -1, -1, -1] and list(slots[:5]) == [32, 33, 34, 35, 36]
    # Growing 7 by 13 tokens: positions 20..32 -> block 1 offsets 4..15, then a new block 3.
    assert lib.kv_seq_extend(h, 7, 13, row, 4, ctypes.byref(ln), slots) == 0
    assert ln.value == 33 and list(row) == [0, 1, 3, -1]
    assert list(slots[:13]) == [16 + o for o in range(4, 16)] + [48]
    # A stale length, a table too short, more blocks than are free: errors that change nothing.
    bad = ctypes.c_int(5)
    assert lib.kv_seq_extend(h, 7, 1, row, 4, ctypes.byref(bad), slots) == 1
    assert lib.kv_seq_extend(h, 7, 200, row, 4, ctypes.byref(ln), slots) == 1
    big = (ctypes.c_int32 * 20)()
    assert lib.kv_seq_extend(h, 8, 200, big, 20, ctypes.byref(ctypes.c_int(0)), (ctypes.c_int32 * 200)()) == 4
    assert ln.value == 33
    # Free 7: blocks 0, 1, 3 go to the back of the queue; a new sequence takes the front (4).
    assert lib.kv_seq_free(h, 7) == 0
    assert lib.kv_seq_free(h, 7) == 9
    ln3 = ctypes.c_int(0)
    assert lib.kv_seq_extend(h, 9, 1, row, 4, ctypes.byref(ln3), slots) == 0
    assert list(row) == [4, -1, -1, -1] and slots[0] == 64
    lib.kv_pool_destroy(h)


def _attn(lib, **kw):
    A = 0x20000000
    args = dict(q=A, k=A, v=A, nb=64, tables=A, max_blocks=8, lens=A, B=4, hq=8, hkv=2, d=64, bs=16,
                dtype=1, scale=0.125, out=A, out_dtype=1, ws=A, ws_bytes=1 << 20, opts=None)
    args.update(kw)
    p = lambda x: ctypes.c_void_p(x) if x else None  # noqa: E731
    return lib.paged_decode_attention(p(args["q"]), p(args["k"]), p(args["v"]), args["nb"], p(args["tables"]),
                                      args["max_blocks"], p(args["lens"]), args["B"], args["hq"], args["hkv"],
                                      args["d"], args["bs"], args["dtype"], args["scale"], p(args["out"]),
                                      args["out_dtype"], p(args["ws"]), args["ws_bytes"], args["opts"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(hq=6, hkv=4), 1),              # not a multiple
    (dict(hq=24, hkv=2), 2),             # group of 12
    (dict(d=96), 2),                     # head_dim
    (dict(bs=512), 2),                   # block size
    (dict(dtype=5), 1),                  # dtype code
    (dict(out_dtype=2), 2),              # f16 in, bf16 out
    (dict(scale=float("inf")), 1),
    (dict(q=0), 1),                      # null pointer
    (dict(k=0x20000008), 1),             # 8-byte aligned cache
    (dict(ws=0x20000010), 1),            # workspace alignment
    (dict(B=-1), 1),
    (dict(dtype=0, out_dtype=0, opts=ctypes.byref(pkv._DecodeOptions(0, 0, 0, 2))), 2),  # fp32 on tensor cores
    (dict(bs=8, opts=ctypes.byref(pkv._DecodeOptions(0, 0, 0, 2))), 2),  # mma needs bs % 16
    (dict(opts=ctypes.byref(pkv._DecodeOptions(0, 0, 16, 0))), 1),       # too many warps
    (dict(opts=ctypes.byref(pkv._DecodeOptions(0, 0, 0, 9))), 1),        # kernel selector
])
def test_attention_argument_validation(lib, kw, code):
    assert _attn(lib, **kw) == code, lib.kv_last_error()


def test_attention_with_no_sequences_is_a_no_op(lib):
    assert _attn(lib, B=0, q=0, out=0) == 0


def test_append_and_slot_mapping_validation(lib):
    assert lib.kv_append(None, 0, None, 1, None, None, None, None) == 1
    assert lib.kv_slot_mapping(None, 4, None, 3, 16, 10, None, None) == 1
    assert lib.kv_slot_mapping(None, 4, None, 0, 16, 10, None, None) == 0
    assert lib.kv_slot_mapping(None, 0, None, 3, 16, 10, None, None) == 1
