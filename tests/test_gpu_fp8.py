"""GPU parity of the FP8 (E4M3) KV cache against the oracle, through the C ABI.

Bars: the quantizing append (plain and fused) bit-exact against the oracle's
codes; attention max |err| <= 2e-3 against the fp64 oracle over the same
codes and scales with fp32 output, plus half an ulp of the output type for
f16/bf16 output.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_slots_gb300 as pkv
from gpu_harness import (LargeCase, SmallCase, attend, attend_append, cache_bits, check_cast, check_output,
                         run_step, scale_opts)
from workloads import SPECS, make_placement, small_spec

pytestmark = pytest.mark.gpu

SCALES = (1.0 / 56.0, 1.0 / 44.0)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _check_all(spec, placement=None, **opts):
    """Plain step (append + attention) and fused step on fresh copies; every output."""
    pl = placement or make_placement(spec)
    case = SmallCase(spec, pl)
    o_slots, kpost, vpost, ref = case.oracle()
    so = scale_opts(spec)
    d = case.device()
    slots, out = run_step(d, spec, pl.num_blocks, out_dtype=torch.float32, **opts)
    outq = attend(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale, **so, **opts)
    assert pkv.device_status() == (0, 0)
    assert np.array_equal(slots.cpu().numpy(), o_slots), "slot mapping"
    assert torch.equal(cache_bits(d["kc"].cpu()), cache_bits(kpost)), "K codes after append"
    assert torch.equal(cache_bits(d["vc"].cpu()), cache_bits(vpost)), "V codes after append"
    e32 = check_output(out, ref, f"{spec.name} fp32 out")
    check_output(outq, ref, f"{spec.name} {spec.dtype} out")
    check_cast(outq, out, spec.name)
    d = case.device()
    out_f, slots_f = attend_append(d["q"], d["kn"], d["vn"], d["kc"], d["vc"], d["tables"], d["ctx"],
                                   spec.attn_scale, seq_ids=d["seq_ids"], out_dtype=torch.float32,
                                   **so, **opts)
    assert pkv.device_status() == (0, 0)
    assert np.array_equal(slots_f.cpu().numpy(), o_slots), "fused slot mapping"
    assert torch.equal(cache_bits(d["kc"].cpu()), cache_bits(kpost)), "K codes after the fused step"
    assert torch.equal(cache_bits(d["vc"].cpu()), cache_bits(vpost)), "V codes after the fused step"
    check_output(out_f, ref, f"{spec.name} fused fp32 out")
    return e32


EDGE_CTX = (1, 15, 16, 17, 31, 32, 33, 0, 100, 257)


@pytest.mark.parametrize("qdtype", ["f16", "bf16"])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_fp8_edge_lengths(qdtype, group):
    spec = small_spec(f"fp8_edge_{qdtype}_{group}", num_q_heads=2 * group, num_kv_heads=2,
                      head_dim=128, block_size=16, dtype=qdtype, seed=70 + group, ctx=EDGE_CTX,
                      kv_dtype="e4m3", kv_scales=SCALES)
    _check_all(spec)


@pytest.mark.parametrize("block_size", [32, 64])
def test_fp8_other_block_sizes(block_size):
    spec = small_spec(f"fp8_bs{block_size}", num_q_heads=16, num_kv_heads=4, head_dim=128,
                      block_size=block_size, dtype="bf16", seed=80 + block_size,
                      ctx=(1, block_size - 1, block_size, block_size + 1, 5 * block_size + 3),
                      kv_dtype="e4m3", kv_scales=(0.0173, 0.0219))
    _check_all(spec)


def test_fp8_llama8b_layer_b8_every_output():
    base = SPECS["llama8b_layer_b8"]
    spec = small_spec("fp8_llama8b_b8", num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                      dtype="bf16", seed=base.seed, ctx=(4096,) * 8, num_blocks=4096,
                      kv_dtype="e4m3", kv_scales=SCALES)
    _check_all(spec)


SPLITS = [
    dict(num_ctas=1), dict(num_ctas=7), dict(num_ctas=300),
    dict(consumer_warps=4), dict(heads_per_stage=2), dict(heads_per_stage=4, consumer_warps=8),
    dict(separate_reduce=True), dict(pdl=False), dict(ctas_per_sm=2), dict(early_reads=True),
]


@pytest.mark.parametrize("opts", SPLITS, ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_fp8_launch_shapes(opts):
    spec = small_spec("fp8_splits", num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                      dtype="bf16", seed=91, ctx=(1, 700, 2049, 33, 0, 4096, 16, 1500),
                      kv_dtype="e4m3", kv_scales=SCALES)
    _check_all(spec, **opts)


def test_fp8_batch32_32_layers_every_sequence():
    """The E4M3 batch-32 step at full size: every sequence of layers 0 and 31,
    the whole layer's codes after the quantizing append bit for bit."""
    spec = SPECS["llama8b_32l_b32_fp8"]
    case = LargeCase(spec, make_placement(spec))
    case.check_layer(0)
    case.check_layer(spec.num_layers - 1, fused=True, early_reads=True)
    del case
    torch.cuda.empty_cache()


def test_fp8_serving_b256_every_sequence():
    """The E4M3 serving step at full size (a 66 GB pool): every sequence of
    layers 0 and 31, the whole layer's codes after the append bit for bit."""
    spec = SPECS["serving_b256_fp8"]
    case = LargeCase(spec, make_placement(spec))
    case.check_layer(0, fused=True, early_reads=True)
    case.check_layer(spec.num_layers - 1)
    del case
    torch.cuda.empty_cache()


def test_fp8_graph_capture_fused():
    spec = small_spec("fp8_graph", num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                      dtype="bf16", seed=93, ctx=(100, 4096, 1, 777), kv_dtype="e4m3", kv_scales=SCALES)
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    _, kpost, vpost, ref = case.oracle()
    d = case.device()
    B, Hq, D = d["q"].shape
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ws = pkv.make_workspace(B, Hq, spec.num_kv_heads, D, "cuda")
    so = scale_opts(spec)
    k0, v0 = d["kc"].clone(), d["vc"].clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.paged_decode_append_attention(d["q"], d["kn"], d["vn"], d["kc"], d["vc"], d["tables"], d["ctx"],
                                          spec.attn_scale, seq_ids=d["seq_ids"], out=out,
                                          out_dtype=torch.float32, workspace=ws, **so)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.paged_decode_append_attention(d["q"], d["kn"], d["vn"], d["kc"], d["vc"], d["tables"], d["ctx"],
                                          spec.attn_scale, seq_ids=d["seq_ids"], out=out,
                                          out_dtype=torch.float32, workspace=ws, **so)
    for _ in range(3):
        d["kc"].copy_(k0)
        d["vc"].copy_(v0)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(cache_bits(d["kc"].cpu()), cache_bits(kpost))
        assert torch.equal(cache_bits(d["vc"].cpu()), cache_bits(vpost))
        check_output(out, ref, "fp8 graph replay")


def test_fp8_argument_checks():
    spec = small_spec("fp8_args", num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                      dtype="bf16", seed=95, ctx=(5, 40), kv_dtype="e4m3", kv_scales=SCALES)
    pl = make_placement(spec)
    d = SmallCase(spec, pl).device()
    q, kc, vc, t, c = d["q"], d["kc"], d["vc"], d["tables"], d["ctx"]
    with pytest.raises(pkv.KVError, match="tensor-core"):
        attend(q, kc, vc, t, c, 0.1, kernel="ffma", **scale_opts(spec))
    with pytest.raises(pkv.KVError) as e:
        attend(q, kc, vc, t, c, 0.1, k_scale=0.0, v_scale=1.0)
    assert e.value.status == 1
    with pytest.raises(pkv.KVError) as e:
        attend(q.float(), kc, vc, t, c, 0.1, **scale_opts(spec))
    assert e.value.status == 2
    # The plain append refuses an E4M3 pool; kv_append_fp8 refuses other pools.
    slots = pkv.slot_mapping(t, c, spec.block_size, pl.num_blocks)
    lib = pkv.load_library()
    st = lib.kv_append(d["pool"]._handle, 0, None, 2, d["kn"].data_ptr(), d["vn"].data_ptr(),
                       slots.data_ptr(), None)
    assert st == 1
    plain = pkv.KVPool(1, 8, 16, 2, 128, "bf16")
    st = lib.kv_append_fp8(plain._handle, 0, None, 2, d["kn"].data_ptr(), d["vn"].data_ptr(), 2,
                           slots.data_ptr(), 1.0, 1.0, None)
    assert st == 1
    assert pkv.device_status() == (0, 0)
