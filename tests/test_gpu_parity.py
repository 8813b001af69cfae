"""GPU parity of the CUDA path against the oracle (runs through the C ABI).

Bars: append and slot mapping bit-exact; attention max |err| <= 2e-3 against
the fp64 oracle with fp32 output, and the same plus half an ulp of the output
type for fp16/bf16 output, which must also be the fp32 output rounded to
nearest even (within one ulp).  Small workloads are checked on every output;
the full-size workloads (in the launch configuration the benchmark times) on
every sequence of the first and last layer (and more), with the whole layer
pool bit-compared after the append.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_slots_gb300 as pkv
from gpu_harness import (LargeCase, SmallCase, attend, attend_append, bits, check_cast, check_output,
                         run_step, sample_sequences)
from workloads import SPECS, make_placement, small_spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _full_small_check(spec, placement=None, kernels=("auto",), **opts):
    pl = placement or make_placement(spec)
    case = SmallCase(spec, pl)
    o_slots, kpost, vpost, ref = case.oracle()
    errs = {}
    for kernel in kernels:
        d = case.device()
        slots, out = run_step(d, spec, pl.num_blocks, out_dtype=torch.float32, kernel=kernel, **opts)
        outq = attend(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"],
                                          spec.attn_scale, kernel=kernel, **opts)
        st, flags = pkv.device_status()
        assert st == 0 and flags == 0, (st, flags)
        assert np.array_equal(slots.cpu().numpy(), o_slots), "slot mapping"
        assert torch.equal(bits(d["kc"].cpu()), bits(kpost)), "K pool after append"
        assert torch.equal(bits(d["vc"].cpu()), bits(vpost)), "V pool after append"
        e32 = check_output(out, ref, f"{spec.name}/{kernel} fp32 out")
        eq = check_output(outq, ref, f"{spec.name}/{kernel} {spec.dtype} out")
        if outq.dtype != torch.float32:
            check_cast(outq, out, f"{spec.name}/{kernel}")
        errs[kernel] = (e32, eq)
        # The same step as one fused call on a fresh copy of the pool.
        d = case.device()
        out_f, slots_f = attend_append(d["q"], d["kn"], d["vn"], d["kc"], d["vc"], d["tables"], d["ctx"],
                                       spec.attn_scale, seq_ids=d["seq_ids"], out_dtype=torch.float32,
                                       kernel=kernel, **opts)
        assert pkv.device_status() == (0, 0)
        assert np.array_equal(slots_f.cpu().numpy(), o_slots), "fused slot mapping"
        assert torch.equal(bits(d["kc"].cpu()), bits(kpost)), "K pool after the fused step"
        assert torch.equal(bits(d["vc"].cpu()), bits(vpost)), "V pool after the fused step"
        check_output(out_f, ref, f"{spec.name}/{kernel} fused fp32 out")
    return errs


def test_tiny_fp32_every_output():
    _full_small_check(SPECS["tiny"], kernels=("auto", "ffma"))


@pytest.mark.parametrize("kernel", ["mma", "ffma"])
def test_llama8b_layer_b8_every_output(kernel):
    _full_small_check(SPECS["llama8b_layer_b8"], kernels=(kernel,))


# Batch independence: a sequence attended alone (a batch of one) against its
# row of the full batch.  The work split hands every CTA an equal share of
# the whole batch's items, so where a sequence's range is cut depends on the
# other sequences, and the partials it is merged from differ; the fp32
# outputs agree to rounding, not bit for bit.
SOLO_ATOL = 1e-5


def test_batch32_32_layers_every_sequence():
    """The batch-32 step at full size (32 layers of 32 x 4096 tokens, the
    bench's launch configuration): every sequence of layers 0 and 31, and the
    whole layer pool after the append bit for bit.  Host memory: two copies
    of a 1 GiB layer; oracle: about 0.5 GB of K/V per layer (well under a
    second on 16 cores)."""
    spec = SPECS["llama8b_32l_b32"]
    case = LargeCase(spec, make_placement(spec))
    case.check_layer(0)
    _, _, out32, _ = case.check_layer(spec.num_layers - 1, fused=True, early_reads=True)
    worst, same = case.solo_agreement(spec.num_layers - 1, [0, 13, 31], out32)
    print(f"batch32 solo: max |diff| {worst:.3e}, bitwise equal {same}/3")
    assert worst <= SOLO_ATOL, worst
    del case
    torch.cuda.empty_cache()


def test_mixed_prefix_b64_every_sequence():
    """The mixed-length prefix-sharing layer at full size: every sequence
    (shared blocks, members that do not append) and the whole pool after the
    append.  Host memory: two copies of a 3.1 GB layer; oracle: about 2 GB of
    K/V (logical), about a second."""
    spec = SPECS["mixed_prefix_b64"]
    pl = make_placement(spec)
    case = LargeCase(spec, pl)
    case.check_layer(0, fused=True)
    # Members of a group that share a table prefix read identical blocks.
    assert (pl.block_tables[0, :8] == pl.block_tables[1, :8]).all()
    del case
    torch.cuda.empty_cache()


def test_serving_b256_every_sequence():
    """The batch-256 serving step at full size (lognormal lengths to 32,768
    tokens, 32 layers, a 131 GB pool): every sequence of four layers (0, 31
    and two seeded ones) with the whole layer pool after the append, then
    every layer on 16 seeded sequences.  Host memory: two copies of a 4.1 GB
    layer; oracle: about 3.7 GB of K/V per whole layer (a second or two) and
    about 0.2 GB per 16-sequence layer."""
    spec = SPECS["serving_b256"]
    case = LargeCase(spec, make_placement(spec))
    rng = np.random.default_rng(44)
    whole = [0, spec.num_layers - 1] + sorted(int(x) for x in rng.choice(np.arange(1, spec.num_layers - 1), 2,
                                                                         replace=False))
    for i, layer in enumerate(whole):
        _, _, out32, _ = case.check_layer(layer, fused=(i % 2 == 0), early_reads=(i % 2 == 0))
    seqs = sample_sequences(case.pl, 16, seed=40)
    worst, same = case.solo_agreement(whole[-1], seqs[:6], out32)
    print(f"serving solo: max |diff| {worst:.3e}, bitwise equal {same}/6")
    assert worst <= SOLO_ATOL, worst
    for layer in range(spec.num_layers):
        if layer not in whole:
            case.check_layer(layer, seqs, fused=True, whole_pool=False, early_reads=True)
    del case
    torch.cuda.empty_cache()


EDGE_CTX = (1, 15, 16, 17, 31, 32, 33, 0, 100)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_edge_lengths_all_shapes(dtype, head_dim, group):
    spec = small_spec(f"edge_{dtype}_{head_dim}_{group}", num_q_heads=2 * group, num_kv_heads=2,
                      head_dim=head_dim, block_size=16, dtype=dtype, seed=head_dim + group,
                      ctx=EDGE_CTX)
    kernels = ("ffma",) if dtype == "f32" else ("mma", "ffma")
    _full_small_check(spec, kernels=kernels)


@pytest.mark.parametrize("block_size", [32, 48, 64])
def test_other_block_sizes(block_size):
    spec = small_spec(f"bs{block_size}", num_q_heads=8, num_kv_heads=2, head_dim=128,
                      block_size=block_size, dtype="bf16", seed=block_size,
                      ctx=(1, block_size - 1, block_size, block_size + 1, 5 * block_size + 3))
    _full_small_check(spec, kernels=("mma", "ffma"))


def test_block_size_8_uses_the_ffma_kernel():
    spec = small_spec("bs8", num_q_heads=4, num_kv_heads=1, head_dim=64, block_size=8, dtype="f16",
                      seed=8, ctx=(1, 7, 8, 9, 70))
    _full_small_check(spec, kernels=("auto", "ffma"))


SPLITS = [dict(), dict(num_ctas=1, consumer_warps=8), dict(num_ctas=2, consumer_warps=1),
          dict(num_ctas=7, consumer_warps=3), dict(num_ctas=64), dict(num_ctas=1000, consumer_warps=15),
          dict(num_ctas=152, consumer_warps=4), dict(heads_per_stage=1), dict(heads_per_stage=2),
          dict(heads_per_stage=4, consumer_warps=12), dict(separate_reduce=True),
          dict(separate_reduce=True, num_ctas=1000), dict(pdl=False), dict(ctas_per_sm=2),
          dict(early_reads=True), dict(early_reads=True, num_ctas=1000, separate_reduce=True)]


@pytest.mark.parametrize("kernel", ["mma", "ffma"])
def test_split_and_warp_counts_agree(kernel):
    """Any grid size, head chunking, warp count or reduce mode gives the same result."""
    spec = small_spec("splits", num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                      dtype="f16", seed=5, ctx=(700, 1, 333, 2048, 16, 45, 0))
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    _, _, _, ref = case.oracle()
    d = case.device()
    slots = pkv.slot_mapping(d["tables"], d["ctx"], spec.block_size, pl.num_blocks)
    d["pool"].append(0, d["kn"], d["vn"], slots, seq_ids=d["seq_ids"])
    outs = []
    for opts in SPLITS:
        out = attend(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                     out_dtype=torch.float32, kernel=kernel, **opts)
        check_output(out, ref, f"{opts}")
        outs.append(out)
    for o, opts in zip(outs[1:], SPLITS[1:]):
        assert torch.max(torch.abs(o - outs[0])).item() <= 2e-5, opts
    assert pkv.device_status() == (0, 0)


def test_workspace_is_reusable_across_calls():
    """The merge counters return to zero: the same workspace serves many calls."""
    spec = small_spec("reuse", num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                      dtype="bf16", seed=6, ctx=(900, 37, 2000))
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    _, _, _, ref = case.oracle()
    d = case.device()
    slots = pkv.slot_mapping(d["tables"], d["ctx"], spec.block_size, pl.num_blocks)
    d["pool"].append(0, d["kn"], d["vn"], slots, seq_ids=d["seq_ids"])
    ws = pkv.make_workspace(3, 8, 2, 128, num_ctas=40)
    for _ in range(5):
        out = torch.full((3, 8, 128), float("nan"), device="cuda")
        pkv.paged_decode_attention(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                                   out=out, out_dtype=torch.float32, workspace=ws, num_ctas=40)
        check_output(out, ref, "reused workspace")
    assert int(ws[:3 * 2 * 4].view(torch.int32).abs().sum().item()) == 0


@pytest.mark.parametrize("num_ctas", [40, 152])
def test_split_merge_is_bitwise_reproducible(num_ctas):
    """Which warp merges a split sequence depends on timing, and a warp at the
    end of its CTA's range reads the parts through shared memory while any
    other reads them from L2; the output bits must not depend on either.
    40 CTAs: about six parts per sequence (the merge that loads every part in
    one round); 152 CTAs: about twenty (the merge in rounds)."""
    spec = SPECS["llama8b_layer_b8"]
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    _, _, _, ref = case.oracle()
    d = case.device()
    slots = pkv.slot_mapping(d["tables"], d["ctx"], spec.block_size, pl.num_blocks)
    d["pool"].append(0, d["kn"], d["vn"], slots, seq_ids=d["seq_ids"])
    ws = pkv.make_workspace(8, 32, 8, 128, num_ctas=num_ctas)
    outs = []
    for _ in range(6):
        out = torch.full((8, 32, 128), float("nan"), device="cuda")
        pkv.paged_decode_attention(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                                   out=out, out_dtype=torch.float32, workspace=ws, num_ctas=num_ctas)
        outs.append(out)
    check_output(outs[0], ref, f"{num_ctas} CTAs")
    for o in outs[1:]:
        assert torch.equal(bits(o), bits(outs[0]))
    assert pkv.device_status() == (0, 0)


MANY_PARTS = [  # (query heads, KV heads, head_dim, dtype, contexts, CTAs): sequences over 10-50 CTAs
    (8, 1, 128, "bf16", (3000, 2000, 700, 1), 24),
    (8, 4, 128, "bf16", (4000, 900), 40),
    (4, 4, 64, "f16", (5000, 1500, 33), 64),
]


@pytest.mark.parametrize("shape", MANY_PARTS, ids=["G8", "G2", "G1"])
@pytest.mark.parametrize("warps", [0, 1])
def test_merge_of_many_parts(shape, warps):
    """Sequences split over more than 32/G CTAs take the merge with four
    (max, sum) slots a lane; with one warp per KV head (warps=1 a head) the
    parts are staged through the ring in chunks.  Against the oracle, and
    bit for bit the same over repeated calls."""
    hq, hkv, d, dtype, ctx, ctas = shape
    spec = small_spec(f"many{hq}_{hkv}", num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=16,
                      dtype=dtype, seed=31 + hq + hkv, ctx=ctx)
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    _, _, _, ref = case.oracle()
    d_ = case.device()
    slots = pkv.slot_mapping(d_["tables"], d_["ctx"], spec.block_size, pl.num_blocks)
    d_["pool"].append(0, d_["kn"], d_["vn"], slots, seq_ids=d_["seq_ids"])
    opts = dict(num_ctas=ctas, kernel="mma")
    if warps:
        opts["consumer_warps"] = hkv if hkv <= 8 else 8
    outs = [attend(d_["q"], d_["kc"], d_["vc"], d_["tables"], d_["ctx"], spec.attn_scale,
                   out_dtype=torch.float32, **opts) for _ in range(3)]
    check_output(outs[0], ref, f"{shape} warps={warps}")
    for o in outs[1:]:
        assert torch.equal(bits(o), bits(outs[0]))
    assert pkv.device_status() == (0, 0)


@pytest.mark.parametrize("kernel", ["mma", "ffma"])
def test_block_relabelling_is_bitwise_invariant(kernel):
    spec = small_spec("relabel", num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                      dtype="bf16", seed=9, ctx=(300, 17, 64, 1))
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    d = case.device()
    base = attend(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                                      kernel=kernel)
    perm = torch.randperm(pl.num_blocks, generator=torch.Generator().manual_seed(3))
    kc2, vc2 = torch.empty_like(d["kc"]), torch.empty_like(d["vc"])
    kc2[perm.cuda()] = d["kc"]
    vc2[perm.cuda()] = d["vc"]
    t = torch.from_numpy(pl.block_tables).long()
    t2 = torch.where(t >= 0, perm[t.clamp(min=0)], torch.full_like(t, -1)).int().cuda()
    out = attend(d["q"], kc2, vc2, t2, d["ctx"], spec.attn_scale, kernel=kernel)
    assert torch.equal(bits(out), bits(base))


@pytest.mark.parametrize("kernel", ["mma", "ffma"])
def test_equal_heads_and_shared_tables(kernel):
    spec = small_spec("equal", num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                      dtype="f16", seed=10, ctx=(130, 130, 40))
    pl = make_placement(spec)
    pl.block_tables[1] = pl.block_tables[0]  # sequence 1 reads sequence 0's blocks
    case = SmallCase(spec, pl)
    d = case.device()
    q = d["q"].clone()
    q[:, 1] = q[:, 0]
    q[1] = q[0]
    out = attend(q, d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                                     kernel=kernel)
    assert torch.equal(bits(out[:, 1]), bits(out[:, 0]))
    assert torch.equal(bits(out[1]), bits(out[0]))
    ref = oracle.paged_decode(q.cpu(), case.kpool, case.vpool, pl.block_tables, pl.context_lens,
                              spec.attn_scale)
    check_output(out, ref, "shared tables")


def test_nan_in_unused_slots_does_not_leak():
    """Slots past a sequence's length may hold anything; the output ignores them."""
    spec = small_spec("nan", num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                      dtype="bf16", seed=12, ctx=(5, 17, 33))
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    for s, c in enumerate(pl.context_lens):
        last = pl.block_tables[s, (c - 1) // 16]
        case.kpool[last, :, c % 16 or 16:, :] = float("nan")
        case.vpool[last, :, c % 16 or 16:, :] = float("nan")
    _, _, _, ref = case.oracle()
    for kernel in ("mma", "ffma"):
        d = case.device()
        _, out = run_step(d, spec, pl.num_blocks, out_dtype=torch.float32, kernel=kernel)
        check_output(out, ref, f"NaN-padded blocks ({kernel})")


def test_device_checks_flag_and_continue():
    spec = small_spec("checks", num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                      dtype="f16", seed=13, ctx=(40, 20))
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    d = case.device()
    assert pkv.device_status() == (0, 0)
    bad = d["tables"].clone()
    bad[0, 1] = pl.num_blocks + 5  # outside the pool
    attend(d["q"], d["kc"], d["vc"], bad, d["ctx"], spec.attn_scale)
    st, flags = pkv.device_status()
    assert st == 7 and flags & pkv.FLAG_BAD_BLOCK_ID
    assert pkv.device_status() == (0, 0)  # read and cleared
    slots = torch.tensor([pl.num_blocks * 16 + 3, -1], dtype=torch.int32, device="cuda")
    before = d["kc"].clone()
    d["pool"].append(0, d["kn"], d["vn"], slots)
    st, flags = pkv.device_status()
    assert st == 7 and flags == pkv.FLAG_BAD_SLOT
    assert torch.equal(bits(before), bits(d["kc"]))  # nothing written
    long_ctx = torch.tensor([40, 10_000], dtype=torch.int32, device="cuda")
    attend(d["q"], d["kc"], d["vc"], d["tables"], long_ctx, spec.attn_scale)
    st, flags = pkv.device_status()
    assert st == 7 and flags & pkv.FLAG_BAD_CONTEXT
    # The context stays usable: a clean call afterwards is still exact.
    _full_small_check(spec, pl)


def test_bounded_wait_times_out_cleanly():
    """A stalled producer makes a consumer's bounded wait run out: status, no fault."""
    spec = small_spec("stall", num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                      dtype="bf16", seed=14, ctx=(200, 300))
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    d = case.device()
    attend(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                               num_ctas=1, test_stall=True)
    st, flags = pkv.device_status()
    assert st == 8 and flags & pkv.FLAG_TIMEOUT
    assert pkv.device_status() == (0, 0)
    _full_small_check(spec, pl)


def test_cuda_graph_capture_of_a_step():
    spec = SPECS["llama8b_layer_b8"]
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    _, _, _, ref = case.oracle()
    d = case.device()
    ws = torch.full((pkv.workspace_bytes(8, 32, 8, 128),), 0xFF, dtype=torch.uint8, device="cuda")
    pkv.workspace_init(ws, 8, 8)
    out = torch.full((8, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
    slots = torch.empty(8, dtype=torch.int32, device="cuda")
    # Warm-up outside the capture (loads the kernels, sets their attributes).
    pkv.slot_mapping(d["tables"], d["ctx"], 16, pl.num_blocks, out=slots)
    pkv.paged_decode_attention(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                               out=out, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pkv.slot_mapping(d["tables"], d["ctx"], 16, pl.num_blocks, out=slots)
            d["pool"].append(0, d["kn"], d["vn"], slots, seq_ids=d["seq_ids"])
            pkv.paged_decode_attention(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                                       out=out, out_dtype=torch.float32, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    check_output(out, ref, "graph replay")
    g.replay()  # appending the same rows again is idempotent
    torch.cuda.synchronize()
    check_output(out, ref, "second replay")


def test_cuda_graph_capture_of_a_fused_step():
    spec = SPECS["llama8b_layer_b8"]
    pl = make_placement(spec)
    case = SmallCase(spec, pl)
    o_slots, kpost, vpost, ref = case.oracle()
    d = case.device()
    ws = torch.full((pkv.workspace_bytes(8, 32, 8, 128),), 0xFF, dtype=torch.uint8, device="cuda")
    pkv.workspace_init(ws, 8, 8)
    out = torch.full((8, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
    slots = torch.full((8,), -7, dtype=torch.int32, device="cuda")

    def step():
        pkv.paged_decode_append_attention(d["q"], d["kn"], d["vn"], d["kc"], d["vc"], d["tables"], d["ctx"],
                                          spec.attn_scale, seq_ids=d["seq_ids"], out=out,
                                          out_dtype=torch.float32, slot_mapping=slots, workspace=ws)

    step()  # warm-up outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    out.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    check_output(out, ref, "fused graph replay")
    assert np.array_equal(slots.cpu().numpy(), o_slots)
    assert torch.equal(bits(d["kc"].cpu()), bits(kpost)) and torch.equal(bits(d["vc"].cpu()), bits(vpost))
