"""The entry point that allocates nothing: paged_decode_attention_static.

Some callers cannot allocate device memory at the moment they run attention:
a serving engine that handed all free device memory to its KV-block pool at
start-up, or code that is given only the tensors it works on (a plugin
inside another framework, whose allocator it may not call).
paged_decode_attention_static serves them from a fixed 8 MiB scratch array
inside the library.  These tests call it through the C ABI twice in a row
and check each result bit for bit against paged_decode_attention with a
caller-provided workspace (same options and grid), and against the oracle.
They also check that the second call changes the free device memory by
nothing, that the largest batch the array holds runs, and that a batch one
sequence larger is refused before anything runs.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_slots_gb300 as pkv
from gpu_harness import SmallCase, bits, check_output
from workloads import SPECS, make_placement, small_spec

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 << 20  # the array's size, as include/pkv.h states it


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _static_vs_workspace(spec, pl, calls=2):
    """Attention of `spec` through the static entry point (`calls` calls in a
    row) against the workspace entry point and the oracle."""
    case = SmallCase(spec, pl)
    d = case.device()
    ref = oracle.paged_decode(case.q, case.kpool, case.vpool, pl.block_tables, pl.context_lens,
                              spec.attn_scale)
    B, Hq, D = d["q"].shape
    ws_out = pkv.paged_decode_attention(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                                        out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_output(ws_out, ref, f"{spec.name} workspace entry point")
    for call in range(calls):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        pkv.paged_decode_attention_static(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"],
                                          spec.attn_scale, out=out, out_dtype=torch.float32)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert pkv.device_status() == (0, 0)
        # Same kernel, same grid, same split: the merge's arithmetic does not
        # depend on which warp merges, so the bits agree.
        assert torch.equal(bits(out), bits(ws_out)), f"call {call}: static and workspace outputs differ"
        check_output(out, ref, f"{spec.name} static entry point, call {call}")
        if call >= 1:  # the first call may load the library's device code; later ones allocate nothing
            assert free_after == free_before, (free_before, free_after)


def test_static_scratch_matches_the_workspace_entry_point():
    spec = SPECS["llama8b_layer_b8"]
    _static_vs_workspace(spec, make_placement(spec))


def _largest_batch_in_the_array(num_q_heads, num_kv_heads, head_dim):
    n = 1
    while pkv.workspace_bytes(n + 1, num_q_heads, num_kv_heads, head_dim) <= STATIC_SCRATCH_BYTES:
        n += 1
    return n


def test_static_scratch_at_its_limit():
    """The largest batch whose scratch fits the array (about 350 sequences of
    the 8B shape on a 152-SM GPU) runs and agrees with the workspace call."""
    hq, hkv, d = 32, 8, 128
    n = _largest_batch_in_the_array(hq, hkv, d)
    assert pkv.workspace_bytes(n, hq, hkv, d) <= STATIC_SCRATCH_BYTES < pkv.workspace_bytes(n + 1, hq, hkv, d)
    rng = np.random.default_rng(71)
    ctx = tuple(int(c) for c in rng.integers(1, 200, size=n))
    spec = small_spec("static_limit", num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=16,
                      dtype="f16", seed=72, ctx=ctx)
    _static_vs_workspace(spec, make_placement(spec))


def test_static_scratch_refuses_sizes_beyond_its_array():
    """One sequence more than the array holds: refused with
    KV_ERR_WORKSPACE_TOO_SMALL, and nothing is launched (the output keeps its
    NaN fill).  Every buffer matches the sizes the call is given, so the
    call would be well formed if the array were larger."""
    hq, hkv, d, bs = 32, 8, 128, 16
    n = _largest_batch_in_the_array(hq, hkv, d) + 1
    q = torch.randn((n, hq, d), device="cuda").half()
    kc = torch.randn((64, hkv, bs, d), device="cuda").half()
    vc = torch.randn_like(kc)
    tables = torch.randint(0, 64, (n, 4), dtype=torch.int32, device="cuda")
    ctx = torch.full((n,), 40, dtype=torch.int32, device="cuda")
    out = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    lib = pkv.load_library()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    torch.cuda.synchronize()
    st = lib.paged_decode_attention_static(
        p(q), p(kc), p(vc), kc.shape[0], p(tables), tables.shape[1], p(ctx), n, hq, hkv, d, bs, pkv.KV_F16,
        1.0 / d ** 0.5, p(out), pkv.KV_F32, None, None)
    assert st == 5, lib.kv_status_string(st)  # KV_ERR_WORKSPACE_TOO_SMALL
    assert b"static scratch" in lib.kv_last_error()
    torch.cuda.synchronize()
    assert bool(torch.isnan(out).all())
    assert pkv.device_status() == (0, 0)
