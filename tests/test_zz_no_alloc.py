"""The entry point that allocates nothing: paged_decode_attention_static.

Some callers cannot allocate device memory -- an engine that handed all free
device memory to its KV-block pool at start-up, or code that is given only
the tensors it works on.  paged_decode_attention_static serves them from a
fixed scratch array inside the library.  These tests call it through the C
ABI twice in a row and compare each result with paged_decode_attention run
with a caller-provided workspace, check that the second call changes the
free device memory by nothing, and that sizes beyond the array are refused
before anything runs.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_slots_gb300 as pkv
from gpu_harness import ATOL, SmallCase
from workloads import SPECS, make_placement

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_static_scratch_matches_the_workspace_entry_point():
    spec = SPECS["llama8b_layer_b8"]
    pl = make_placement(spec)
    d = SmallCase(spec, pl).device()
    B, Hq, D = d["q"].shape
    ref = pkv.paged_decode_attention(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                                     out_dtype=torch.float32)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        pkv.paged_decode_attention_static(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"],
                                          spec.attn_scale, out=out, out_dtype=torch.float32)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert pkv.device_status() == (0, 0)
        assert bool(torch.isfinite(out).all())
        diff = (out - ref).abs().max().item()
        assert diff <= ATOL, f"call {call}: max |static - workspace| = {diff:.3e}"
        if call == 1:  # the first call may load the library's device code; the second allocates nothing
            assert free_after == free_before, (free_before, free_after)


def test_static_scratch_refuses_sizes_beyond_its_array():
    spec = SPECS["llama8b_layer_b8"]
    pl = make_placement(spec)
    d = SmallCase(spec, pl).device()
    lib = pkv.load_library()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    # 100,000 sequences need far more than the 8 MiB array; nothing is read
    # or launched, validation stops the call first.
    st = lib.paged_decode_attention_static(
        p(d["q"]), p(d["kc"]), p(d["vc"]), pl.num_blocks, p(d["tables"]), pl.block_tables.shape[1],
        p(d["ctx"]), 100_000, 32, 8, 128, 16, pkv.KV_F16, spec.attn_scale, p(d["q"]), pkv.KV_F32, None,
        None)
    assert st == 5, lib.kv_status_string(st)  # KV_ERR_WORKSPACE_TOO_SMALL
    assert b"workspace" in lib.kv_last_error()
