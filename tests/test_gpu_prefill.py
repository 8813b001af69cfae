"""GPU parity of multi-token queries (chunked prefill) against the oracle.

Bars: the varlen slot mapping and the append of every new token bit-exact;
attention max |err| <= 2e-3 against the fp64 oracle with fp32 output, plus
half an ulp of the output type for f16/bf16 output.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_slots_gb300 as pkv
from gpu_harness import bits, check_cast, check_output, compact_blocks, take
from workloads import (SPECS, fill_pool_layer, make_placement, new_token_counts, pool_layer_values, small_spec,
                       step_token_values)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _step(spec, nq, out_dtype=torch.float32, check_pool=True, scale=None):
    """Slot mapping, append and causal attention of one multi-token step,
    through the library and through the oracle; every output compared."""
    scale = spec.attn_scale if scale is None else scale
    pl = make_placement(spec)
    ctx = pl.context_lens
    nq = np.asarray(nq, np.int32)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    T = int(qs[-1])
    k_pre, v_pre = pool_layer_values(spec, pl.num_blocks, 0, "cpu")
    q, kn, vn = step_token_values(spec, T, 0, "cpu")
    o_slots = oracle.slot_mapping_varlen(pl.block_tables, qs, ctx, spec.block_size)
    k_post, v_post = oracle.append(k_pre, v_pre, kn, vn, o_slots)
    ref = oracle.paged_prefill(q, k_post, v_post, pl.block_tables, qs, ctx, scale)

    pool = pkv.KVPool(1, pl.num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim, spec.torch_dtype)
    kc, vc = pool.layer(0)
    kc.copy_(k_pre)
    vc.copy_(v_pre)
    tables = torch.from_numpy(pl.block_tables).cuda()
    ctx_d = torch.from_numpy(ctx).cuda()
    qs_d = torch.from_numpy(qs).cuda()
    slots = pkv.slot_mapping_varlen(tables, qs_d, ctx_d, spec.block_size, pl.num_blocks, num_tokens=T)
    pool.append(0, kn.cuda(), vn.cuda(), slots)
    out = torch.full((T, spec.num_q_heads, spec.head_dim), float("nan"), dtype=out_dtype, device="cuda")
    pkv.paged_prefill_attention(q.cuda(), kc, vc, tables, qs_d, ctx_d, scale, out=out,
                                out_dtype=out_dtype)
    assert pkv.device_status() == (0, 0)
    assert np.array_equal(slots.cpu().numpy(), o_slots), "varlen slot mapping"
    if check_pool:
        assert torch.equal(bits(kc.cpu()), bits(k_post)) and torch.equal(bits(vc.cpu()), bits(v_post))
    if out_dtype != torch.float32:
        # The same attention with fp32 output: the q-dtype output is it rounded to nearest even.
        out32 = torch.full_like(out, float("nan"), dtype=torch.float32)
        pkv.paged_prefill_attention(q.cuda(), kc, vc, tables, qs_d, ctx_d, scale, out=out32,
                                    out_dtype=torch.float32)
        check_output(out32, ref, f"{spec.name} prefill fp32")
        check_cast(out, out32, f"{spec.name} prefill")
    return check_output(out, ref, f"{spec.name} prefill {out_dtype}")


CTX = (1, 15, 16, 17, 33, 64, 100, 257, 40)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_mixed_step_all_shapes(dtype, head_dim, group):
    spec = small_spec(f"prefill_{dtype}_{head_dim}_{group}", num_q_heads=2 * group, num_kv_heads=2,
                      head_dim=head_dim, block_size=16, dtype=dtype, seed=100 + head_dim + group, ctx=CTX)
    nq = new_token_counts(CTX, seed=group, max_chunk=70)
    nq[-1] = CTX[-1]  # one whole prompt (no earlier context)
    _step(spec, nq)


@pytest.mark.parametrize("block_size", [32, 64, 128])
def test_other_block_sizes(block_size):
    ctx = (1, block_size - 1, block_size + 1, 3 * block_size + 5, 200)
    spec = small_spec(f"prefill_bs{block_size}", num_q_heads=8, num_kv_heads=2, head_dim=128,
                      block_size=block_size, dtype="bf16", seed=block_size, ctx=ctx)
    _step(spec, new_token_counts(ctx, seed=3, max_chunk=150))


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.3])
def test_negative_zero_and_large_scale(head_dim, scale):
    # A negative scale favours the keys least aligned with q; a zero scale
    # gives the mean of V over each token's visible keys.
    ctx = (1, 40, 130, 77)
    spec = small_spec(f"prefill_scale_{head_dim}", num_q_heads=8, num_kv_heads=2, head_dim=head_dim,
                      block_size=16, dtype="bf16", seed=21, ctx=ctx)
    _step(spec, [1, 40, 65, 3], scale=scale)


@pytest.mark.parametrize("block_size", [32, 64, 128])
@pytest.mark.parametrize("group", [1, 2, 8])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tensor_core_block_sizes_and_groups(block_size, group, dtype):
    # The tcgen05 kernel's two loaders (per-lane copies below 64-token blocks,
    # TMA boxes from 64 up) with every query-head group size; contexts cross
    # block and 64-key tile boundaries and end mid-block.
    ctx = (1, block_size + 3, 129, 2 * block_size + 64 + 7, 300)
    spec = small_spec(f"prefill_tc_bs{block_size}_g{group}_{dtype}", num_q_heads=2 * group, num_kv_heads=2,
                      head_dim=128, block_size=block_size, dtype=dtype, seed=31 + block_size + group, ctx=ctx)
    _step(spec, new_token_counts(ctx, seed=group, max_chunk=200))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_output_in_input_dtype(dtype, head_dim):
    spec = small_spec(f"prefill_out_{dtype}_{head_dim}", num_q_heads=32, num_kv_heads=8, head_dim=head_dim,
                      block_size=16, dtype=dtype, seed=7, ctx=(300, 17, 1, 64))
    _step(spec, [70, 17, 1, 5], out_dtype=spec.torch_dtype)


def test_long_chunk_after_context():
    # A 2048-token chunk after 2048 tokens of earlier context, next to decodes:
    # the shape of a chunked-prefill step of the Llama-3-8B-shaped layer.
    spec = small_spec("prefill_long", num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                      dtype="bf16", seed=9, ctx=(4096, 700, 33, 4096))
    _step(spec, [2048, 1, 1, 1])


def test_chunked_prompt_equals_one_step():
    # A 300-token prompt processed in chunks of 128, 128, 44 gives the rows of
    # the prompt processed at once (same cache contents).
    spec = small_spec("prefill_chunks", num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                      dtype="f16", seed=11, ctx=(300,))
    pl = make_placement(spec)
    k_pre, _ = pool_layer_values(spec, pl.num_blocks, 0, "cuda")
    v_pre = torch.randn_like(k_pre.float()).to(k_pre.dtype)
    q, _, _ = step_token_values(spec, 300, 0, "cuda")
    tables = torch.from_numpy(pl.block_tables).cuda()
    whole = pkv.paged_prefill_attention(q, k_pre, v_pre, tables, torch.tensor([0, 300], dtype=torch.int32,
                                        device="cuda"), torch.tensor([300], dtype=torch.int32, device="cuda"),
                                        spec.attn_scale, out_dtype=torch.float32)
    done = 0
    for n in (128, 128, 44):
        part = pkv.paged_prefill_attention(q[done:done + n].contiguous(), k_pre, v_pre, tables,
                                           torch.tensor([0, n], dtype=torch.int32, device="cuda"),
                                           torch.tensor([done + n], dtype=torch.int32, device="cuda"),
                                           spec.attn_scale, out_dtype=torch.float32)
        assert torch.equal(part, whole[done:done + n]), f"chunk at {done}"
        done += n


def test_bad_lengths_flagged_and_skipped():
    spec = small_spec("prefill_bad", num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                      dtype="f16", seed=13, ctx=(20, 5))
    pl = make_placement(spec)
    k_pre, v_pre = pool_layer_values(spec, pl.num_blocks, 0, "cuda")
    q, _, _ = step_token_values(spec, 12, 0, "cuda")
    tables = torch.from_numpy(pl.block_tables).cuda()
    qs = torch.tensor([0, 4, 12], dtype=torch.int32, device="cuda")  # second: 8 new tokens > 5 cached
    ctx = torch.tensor([20, 5], dtype=torch.int32, device="cuda")
    out = torch.full((12, 4, 64), 7.0, dtype=torch.float32, device="cuda")
    pkv.paged_prefill_attention(q, k_pre, v_pre, tables, qs, ctx, spec.attn_scale, out=out,
                                out_dtype=torch.float32)
    st, flags = pkv.device_status()
    assert flags & pkv.FLAG_BAD_CONTEXT and st != 0
    assert torch.all(out[4:] == 7.0)  # the bad sequence's rows are not written
    assert torch.isfinite(out[:4]).all()
    with pytest.raises(pkv.KVError):  # f16 needs blocks of a multiple of 16 tokens
        pkv.paged_prefill_attention(q, k_pre.view(-1, 2, 8, 64).contiguous(), v_pre.view(-1, 2, 8, 64).contiguous(),
                                    tables, qs, ctx, 0.1)


def test_chunked_prefill_b32_full_size_sampled():
    # Layer 0 of the benchmarked step at full size (16,384 new tokens: 32 decodes
    # at 4096 tokens of context and a 16,352-token chunk after 16,384 cached
    # tokens), run by the library in one call.  The oracle recomputes sampled
    # tokens, each as one query over its causal prefix, from the seeded
    # pre-append pool and its own append of every new token of the sampled
    # sequences.
    spec = SPECS["chunked_prefill_b32"]
    pl = make_placement(spec)
    ctx = pl.context_lens
    nq = np.asarray(spec.new_tokens, np.int32)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    T = int(qs[-1])
    pool = pkv.KVPool(1, pl.num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim, spec.torch_dtype)
    kc, vc = pool.layer(0)
    fill_pool_layer(spec, 0, kc, vc)
    q, kn, vn = step_token_values(spec, T, 0, "cuda")
    long_s = int(np.argmax(nq))
    seqs = [0, 17, long_s]
    used, ctab = compact_blocks(pl.block_tables, seqs)
    used_t = torch.from_numpy(used.astype(np.int64)).cuda()
    k_pre, v_pre = take(kc, used_t).cpu(), take(vc, used_t).cpu()  # the oracle's pool: pre-append
    tables = torch.from_numpy(pl.block_tables).cuda()
    ctx_d = torch.from_numpy(ctx).cuda()
    qs_d = torch.from_numpy(qs).cuda()
    slots = pkv.slot_mapping_varlen(tables, qs_d, ctx_d, spec.block_size, pl.num_blocks, num_tokens=T)
    pool.append(0, kn, vn, slots)
    out = torch.full((T, spec.num_q_heads, spec.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_prefill_attention(q, kc, vc, tables, qs_d, ctx_d, spec.attn_scale, out=out, out_dtype=torch.float32)
    assert pkv.device_status() == (0, 0)
    # The oracle's append of every new token of the sampled sequences.
    nq_s = nq[seqs]
    qs_s = np.concatenate([[0], np.cumsum(nq_s)]).astype(np.int32)
    rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in seqs])
    rows_t = torch.from_numpy(rows).cuda()
    o_slots = oracle.slot_mapping_varlen(ctab, qs_s, ctx[seqs], spec.block_size)
    k_post, v_post = oracle.append(k_pre, v_pre, kn[rows_t].cpu(), vn[rows_t].cpu(), o_slots)
    assert torch.equal(bits(take(kc, used_t).cpu()), bits(k_post)), "K blocks after the append"
    assert torch.equal(bits(take(vc, used_t).cpu()), bits(v_post)), "V blocks after the append"
    # Sampled tokens: both decodes, and the chunk's first, last and three inner tokens.
    picks = [(0, 0), (1, 0)] + [(2, i) for i in (0, 1, 4095, 8190, int(nq[long_s]) - 1)]
    for k, i in picks:
        s = seqs[k]
        pos = int(ctx[s] - nq[s] + i)
        t = int(qs[s] + i)
        ref = oracle.paged_decode(q[t:t + 1].cpu(), k_post, v_post, ctab[k:k + 1],
                                  np.array([pos + 1], np.int32), spec.attn_scale)
        check_output(out[t:t + 1], ref, f"chunked_prefill_b32 sequence {s} token {i} (position {pos})")


# ------------------------------------------------------------ f32 and E4M3
F32_CTX = (1, 15, 16, 17, 40, 100, 33)


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("block_size", [8, 16, 48])
def test_f32_multi_token_queries(head_dim, group, block_size):
    """f32 q and cache (the CUDA-core kernel, any block size): every output."""
    spec = small_spec(f"prefill_f32_{head_dim}_{group}_{block_size}", num_q_heads=2 * group, num_kv_heads=2,
                      head_dim=head_dim, block_size=block_size, dtype="f32", seed=200 + head_dim + group + block_size,
                      ctx=F32_CTX)
    nq = new_token_counts(F32_CTX, seed=group, max_chunk=40)
    nq[3] = F32_CTX[3]  # one whole prompt
    _step(spec, nq)


def _step_fp8(spec, nq, out_dtype=torch.float32, scale=None):
    """The multi-token step over an E4M3 cache: varlen slots, the quantizing
    append of every new token (codes bit-exact) and the causal attention over
    the codes times the scales, against the oracle."""
    scale = spec.attn_scale if scale is None else scale
    ks, vs = spec.kv_scales
    pl = make_placement(spec)
    ctx = pl.context_lens
    nq = np.asarray(nq, np.int32)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    T = int(qs[-1])
    k_pre, v_pre = pool_layer_values(spec, pl.num_blocks, 0, "cpu")
    q, kn, vn = step_token_values(spec, T, 0, "cpu")
    o_slots = oracle.slot_mapping_varlen(pl.block_tables, qs, ctx, spec.block_size)
    k_post, v_post = oracle.append_e4m3(k_pre, v_pre, kn, vn, o_slots, ks, vs)
    ref = oracle.paged_prefill(q, k_post, v_post, pl.block_tables, qs, ctx, scale, k_scale=ks, v_scale=vs)
    pool = pkv.KVPool(1, pl.num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim, torch.float8_e4m3fn)
    kc, vc = pool.layer(0)
    kc.view(torch.uint8).copy_(k_pre.view(torch.uint8))
    vc.view(torch.uint8).copy_(v_pre.view(torch.uint8))
    tables = torch.from_numpy(pl.block_tables).cuda()
    ctx_d = torch.from_numpy(ctx).cuda()
    qs_d = torch.from_numpy(qs).cuda()
    slots = pkv.slot_mapping_varlen(tables, qs_d, ctx_d, spec.block_size, pl.num_blocks, num_tokens=T)
    pool.append(0, kn.cuda(), vn.cuda(), slots, k_scale=ks, v_scale=vs)
    out = torch.full((T, spec.num_q_heads, spec.head_dim), float("nan"), dtype=out_dtype, device="cuda")
    pkv.paged_prefill_attention(q.cuda(), kc, vc, tables, qs_d, ctx_d, scale, out=out, out_dtype=out_dtype,
                                k_scale=ks, v_scale=vs)
    assert pkv.device_status() == (0, 0)
    assert np.array_equal(slots.cpu().numpy(), o_slots), "varlen slot mapping"
    assert torch.equal(kc.view(torch.uint8).cpu(), k_post.view(torch.uint8)), "K codes after the append"
    assert torch.equal(vc.view(torch.uint8).cpu(), v_post.view(torch.uint8)), "V codes after the append"
    if out_dtype != torch.float32:
        out32 = torch.full_like(out, float("nan"), dtype=torch.float32)
        pkv.paged_prefill_attention(q.cuda(), kc, vc, tables, qs_d, ctx_d, scale, out=out32,
                                    out_dtype=torch.float32, k_scale=ks, v_scale=vs)
        check_output(out32, ref, f"{spec.name} E4M3 prefill fp32")
        check_cast(out, out32, f"{spec.name} E4M3 prefill")
    return check_output(out, ref, f"{spec.name} E4M3 prefill {out_dtype}")


FP8_SCALES = (1.0 / 56.0, 1.0 / 44.0)
FP8_CTX = (1, 15, 16, 17, 33, 64, 100, 257, 40)


@pytest.mark.parametrize("qdtype", ["f16", "bf16"])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_fp8_multi_token_queries(qdtype, group):
    spec = small_spec(f"prefill_fp8_{qdtype}_{group}", num_q_heads=2 * group, num_kv_heads=2, head_dim=128,
                      block_size=16, dtype=qdtype, seed=300 + group, ctx=FP8_CTX, kv_dtype="e4m3",
                      kv_scales=FP8_SCALES)
    nq = new_token_counts(FP8_CTX, seed=group, max_chunk=70)
    nq[-1] = FP8_CTX[-1]  # one whole prompt
    _step_fp8(spec, nq)


@pytest.mark.parametrize("block_size", [32, 64, 128])
def test_fp8_multi_token_block_sizes_and_output_type(block_size):
    ctx = (1, block_size - 1, block_size + 1, 3 * block_size + 5, 200)
    spec = small_spec(f"prefill_fp8_bs{block_size}", num_q_heads=8, num_kv_heads=2, head_dim=128,
                      block_size=block_size, dtype="bf16", seed=310 + block_size, ctx=ctx, kv_dtype="e4m3",
                      kv_scales=(0.0173, 0.0219))
    _step_fp8(spec, new_token_counts(ctx, seed=5, max_chunk=150), out_dtype=torch.bfloat16)


def test_fp8_long_chunk_and_negative_scale():
    # A 700-token chunk after 2,000 cached tokens next to decodes, the 8B
    # head shape; and a negative scale over the same cache.
    spec = small_spec("prefill_fp8_long", num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                      dtype="bf16", seed=321, ctx=(2700, 40, 1, 900), kv_dtype="e4m3", kv_scales=FP8_SCALES)
    _step_fp8(spec, [700, 1, 1, 1])
    _step_fp8(spec, [700, 1, 1, 1], scale=-0.05)
