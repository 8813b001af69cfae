"""Seeded synthetic inputs for one paged-KV decode step.

This module is shared by the oracle-side tests and by the CUDA side (tests,
bench, smoke).  It holds random draws and block placement only: which
physical blocks each sequence owns, how long each sequence is, and the
N(0, 1) values of q, the new K/V rows and the pool.  It contains none of the
method's arithmetic (no slot formula, no scatter, no attention).

Workload shapes follow the pages' running example: a Llama-3-8B-shaped
attention layer (32 query heads, 8 KV heads, head_dim 128, 16-token blocks)
from "vLLM Architecture and Installation", Example 6, decoding 4096-token
contexts at batch 8..32 as in "Batching and Scheduling", Example 1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
                "e4m3": torch.float8_e4m3fn}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}


@dataclass(frozen=True)
class WorkloadSpec:
    """Shape and distribution of one synthetic decode step."""

    name: str
    num_layers: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str  # "f32" | "f16" | "bf16" (q, K, V and the pool share it)
    seed: int
    ctx_dist: str  # "list" | "const" | "uniform" | "lognormal"
    ctx_list: tuple = ()
    ctx_const: int = 0
    ctx_max: int = 0
    lognormal_median: float = 0.0
    lognormal_sigma: float = 1.0
    num_blocks: int = 0  # 0: derived from the placement rule below
    pool_rule: str = "fixed"  # "fixed" | "twice_used" | "ninety_percent_used"
    prefix_tokens: int = 0  # >0: groups of `prefix_group` sequences share this prefix
    prefix_group: int = 8
    scale: float = 0.0  # 0: 1/sqrt(head_dim)
    # Cache storage type when it differs from `dtype` ("e4m3": an FP8 cache
    # whose codes stand for kv_scales[0] (K) and kv_scales[1] (V) times their
    # values; q and the new rows stay in `dtype`).
    kv_dtype: str = ""
    kv_scales: tuple = (1.0, 1.0)
    # New tokens per sequence for a multi-token (chunked-prefill) step; empty:
    # a decode step (one new token each).
    new_tokens: tuple = ()

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def attn_scale(self) -> float:
        return self.scale if self.scale else 1.0 / math.sqrt(self.head_dim)

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.dtype]

    @property
    def cache_dtype(self) -> str:
        return self.kv_dtype or self.dtype

    @property
    def cache_torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.cache_dtype]

    @property
    def cache_elem_bytes(self) -> int:
        return ELEM_BYTES[self.cache_dtype]

    @property
    def fp8(self) -> bool:
        return self.cache_dtype == "e4m3"


SPECS = {
    # 1 layer, 4 sequences, fp32, 64-block pool with permuted tables.
    "tiny": WorkloadSpec(
        name="tiny", num_layers=1, num_seqs=4, num_q_heads=8, num_kv_heads=2,
        head_dim=64, block_size=16, dtype="f32", seed=0, ctx_dist="list",
        ctx_list=(17, 64, 100, 256), num_blocks=64, scale=1.0 / 8.0),
    # One Llama-3-8B-shaped layer, batch 8 x 4096, fp16, 4096-block pool.
    "llama8b_layer_b8": WorkloadSpec(
        name="llama8b_layer_b8", num_layers=1, num_seqs=8, num_q_heads=32,
        num_kv_heads=8, head_dim=128, block_size=16, dtype="f16", seed=1,
        ctx_dist="const", ctx_const=4096, num_blocks=4096),
    # Same shape, batch 32 x 4096, 32 layers back to back, bf16.
    "llama8b_32l_b32": WorkloadSpec(
        name="llama8b_32l_b32", num_layers=32, num_seqs=32, num_q_heads=32,
        num_kv_heads=8, head_dim=128, block_size=16, dtype="bf16", seed=2,
        ctx_dist="const", ctx_const=4096, pool_rule="twice_used"),
    # Batch 64, lengths U[1, 16384], 2048-token prefix shared by groups of 8.
    "mixed_prefix_b64": WorkloadSpec(
        name="mixed_prefix_b64", num_layers=1, num_seqs=64, num_q_heads=32,
        num_kv_heads=8, head_dim=128, block_size=16, dtype="f16", seed=3,
        ctx_dist="uniform", ctx_max=16384, pool_rule="twice_used",
        prefix_tokens=2048, prefix_group=8),
    # Batch 256, lognormal lengths (median 2048, capped at 32768), 32 layers,
    # bf16, 32-token blocks, pool sized so that 10 % of its blocks stay free.
    "serving_b256": WorkloadSpec(
        name="serving_b256", num_layers=32, num_seqs=256, num_q_heads=32,
        num_kv_heads=8, head_dim=128, block_size=32, dtype="bf16", seed=4,
        ctx_dist="lognormal", lognormal_median=2048.0, lognormal_sigma=1.0,
        ctx_max=32768, pool_rule="ninety_percent_used"),
    # The batch-32 step with an FP8 (E4M3) cache: K codes ~ N(0, 56^2) and V
    # codes ~ N(0, 44^2) rounded to E4M3, scales 1/56 and 1/44, so the cached
    # values are N(0, 1) draws at E4M3 precision.
    "llama8b_32l_b32_fp8": WorkloadSpec(
        name="llama8b_32l_b32_fp8", num_layers=32, num_seqs=32, num_q_heads=32,
        num_kv_heads=8, head_dim=128, block_size=16, dtype="bf16", seed=2,
        ctx_dist="const", ctx_const=4096, pool_rule="twice_used",
        kv_dtype="e4m3", kv_scales=(1.0 / 56.0, 1.0 / 44.0)),
    # A chunked-prefill step at the token budget the pages list for GPUs with
    # 160 GiB or more (16,384 tokens): 32 decodes at 4096 tokens of context
    # and a 16,352-token chunk continuing a prompt after 16,384 cached tokens.
    "chunked_prefill_b32": WorkloadSpec(
        name="chunked_prefill_b32", num_layers=32, num_seqs=33, num_q_heads=32,
        num_kv_heads=8, head_dim=128, block_size=16, dtype="bf16", seed=5,
        ctx_dist="list", ctx_list=(4096,) * 32 + (32736,), pool_rule="twice_used",
        new_tokens=(1,) * 32 + (16352,)),
    # The serving mix with an FP8 cache (same lengths and placement rule).
    "serving_b256_fp8": WorkloadSpec(
        name="serving_b256_fp8", num_layers=32, num_seqs=256, num_q_heads=32,
        num_kv_heads=8, head_dim=128, block_size=32, dtype="bf16", seed=4,
        ctx_dist="lognormal", lognormal_median=2048.0, lognormal_sigma=1.0,
        ctx_max=32768, pool_rule="ninety_percent_used",
        kv_dtype="e4m3", kv_scales=(1.0 / 56.0, 1.0 / 44.0)),
}


@dataclass
class Placement:
    """Block tables and lengths of one step (host arrays).

    context_lens counts the token appended in this step; block_tables rows list
    physical block ids in logical order, padded with -1.  appends[s] is False
    where the newest position of s falls in a block shared with other
    sequences (that sequence writes nothing this step).
    """

    context_lens: np.ndarray
    block_tables: np.ndarray
    num_blocks: int
    appends: np.ndarray
    used_blocks: int
    unique_kv_tokens: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


def draw_context_lens(spec: WorkloadSpec) -> np.ndarray:
    rng = np.random.default_rng(spec.seed)
    if spec.ctx_dist == "list":
        c = np.array(spec.ctx_list, dtype=np.int64)
    elif spec.ctx_dist == "const":
        c = np.full(spec.num_seqs, spec.ctx_const, dtype=np.int64)
    elif spec.ctx_dist == "uniform":
        c = rng.integers(1, spec.ctx_max + 1, size=spec.num_seqs)
    elif spec.ctx_dist == "lognormal":
        c = np.floor(rng.lognormal(math.log(spec.lognormal_median),
                                   spec.lognormal_sigma, size=spec.num_seqs))
        c = np.clip(c, 1, spec.ctx_max).astype(np.int64)
    else:
        raise ValueError(spec.ctx_dist)
    return c.astype(np.int32)


def make_placement(spec: WorkloadSpec, context_lens=None) -> Placement:
    """Random physical placement of every sequence's blocks.

    Blocks are drawn without replacement from a random permutation of the
    pool.  With a shared prefix, the first prefix_tokens/block_size logical
    blocks of every member of a group point at the same physical blocks.
    """
    ctx = draw_context_lens(spec) if context_lens is None else np.asarray(context_lens, np.int32)
    bs = spec.block_size
    nblk = [(int(c) + bs - 1) // bs for c in ctx]
    B = len(ctx)
    # Per-sequence block demand, with shared prefix blocks counted once per group.
    shared_per_group = {}
    if spec.prefix_tokens:
        pb = spec.prefix_tokens // bs
        for s in range(B):
            gidx = s // spec.prefix_group
            shared_per_group[gidx] = max(shared_per_group.get(gidx, 0), min(pb, nblk[s]))
        private = sum(max(0, n - pb) for n in nblk)
        used = private + sum(shared_per_group.values())
    else:
        pb = 0
        used = sum(nblk)
    if spec.pool_rule == "fixed":
        NB = spec.num_blocks
    elif spec.pool_rule == "twice_used":
        NB = 2 * used
    elif spec.pool_rule == "ninety_percent_used":
        NB = math.ceil(used / 0.9)
    else:
        raise ValueError(spec.pool_rule)
    if used > NB:
        raise ValueError(f"{spec.name}: {used} blocks needed, pool has {NB}")
    rng = np.random.default_rng(spec.seed + 7919)
    perm = rng.permutation(NB).astype(np.int32)
    cursor = 0
    maxb = max(1, max(nblk))
    tables = np.full((B, maxb), -1, dtype=np.int32)
    group_blocks = {}
    for gidx, n in sorted(shared_per_group.items()):
        group_blocks[gidx] = perm[cursor:cursor + n]
        cursor += n
    appends = np.ones(B, dtype=bool)
    for s in range(B):
        n = nblk[s]
        if pb:
            k = min(pb, n)
            tables[s, :k] = group_blocks[s // spec.prefix_group][:k]
            tables[s, k:n] = perm[cursor:cursor + (n - k)]
            cursor += n - k
            # Newest position inside a shared block: nothing is written.
            appends[s] = (int(ctx[s]) - 1) // bs >= pb
        else:
            tables[s, :n] = perm[cursor:cursor + n]
            cursor += n
    appends &= ctx > 0
    unique_tokens = int(ctx.sum())
    if pb:
        unique_tokens = 0
        for gidx in shared_per_group:
            members = [s for s in range(B) if s // spec.prefix_group == gidx]
            unique_tokens += max(min(int(ctx[s]), spec.prefix_tokens) for s in members)
            unique_tokens += sum(max(0, int(ctx[s]) - spec.prefix_tokens) for s in members)
    return Placement(context_lens=ctx.astype(np.int32), block_tables=tables,
                     num_blocks=int(NB), appends=appends, used_blocks=int(used),
                     unique_kv_tokens=unique_tokens)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, dtype, seed, device, chunk_elems=1 << 26) -> torch.Tensor:
    """N(0, 1) in fp32, rounded to `dtype` (round-to-nearest-even), chunked."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    g = _gen(seed, device)
    n = flat.numel()
    for a in range(0, n, chunk_elems):
        b = min(n, a + chunk_elems)
        flat[a:b] = torch.randn(b - a, generator=g, dtype=torch.float32, device=device).to(dtype)
    return out


def value_seed(spec: WorkloadSpec, layer: int, kind: int) -> int:
    return spec.seed * 1_000_003 + layer * 16 + kind


def _sigma(spec: WorkloadSpec, kind: int) -> float:
    """Standard deviation of the stored values: 1, or 1 / scale for E4M3 codes."""
    return 1.0 / spec.kv_scales[kind - 1] if spec.fp8 else 1.0


def pool_layer_values(spec: WorkloadSpec, num_blocks: int, layer: int, device="cpu"):
    """Pre-step contents of one layer's K and V pools: [NB, Hkv, bs, D] each."""
    shape = (num_blocks, spec.num_kv_heads, spec.block_size, spec.head_dim)
    k = torch.empty(shape, dtype=spec.cache_torch_dtype, device=device)
    v = torch.empty(shape, dtype=spec.cache_torch_dtype, device=device)
    fill_pool_layer(spec, layer, k, v)
    return k, v


def fill_pool_layer(spec: WorkloadSpec, layer: int, k_view: torch.Tensor, v_view: torch.Tensor):
    """One layer's pool contents, written into existing [NB, Hkv, bs, D] views:
    N(0, sigma^2) fp32 draws rounded to the cache type by torch's own cast."""
    for view, kind in ((k_view, 1), (v_view, 2)):
        flat = view.reshape(-1)
        g = _gen(value_seed(spec, layer, kind), view.device)
        sigma = _sigma(spec, kind)
        n = flat.numel()
        step = 1 << 26
        for a in range(0, n, step):
            b = min(n, a + step)
            x = torch.randn(b - a, generator=g, dtype=torch.float32, device=view.device)
            if sigma != 1.0:
                x = x * sigma
            flat[a:b] = x.to(view.dtype)


def step_layer_values(spec: WorkloadSpec, num_seqs: int, layer: int, device="cpu"):
    """q [B, Hq, D] and the new token's K, V rows [B, Hkv, D] for one layer."""
    q = _normal((num_seqs, spec.num_q_heads, spec.head_dim), spec.torch_dtype,
                value_seed(spec, layer, 3), device)
    kn = _normal((num_seqs, spec.num_kv_heads, spec.head_dim), spec.torch_dtype,
                 value_seed(spec, layer, 4), device)
    vn = _normal((num_seqs, spec.num_kv_heads, spec.head_dim), spec.torch_dtype,
                 value_seed(spec, layer, 5), device)
    return q, kn, vn


def step_token_values(spec: WorkloadSpec, num_tokens: int, layer: int, device="cpu"):
    """q [T, Hq, D] and the new K, V rows [T, Hkv, D] of a step with T new tokens."""
    q = _normal((num_tokens, spec.num_q_heads, spec.head_dim), spec.torch_dtype,
                value_seed(spec, layer, 6), device)
    kn = _normal((num_tokens, spec.num_kv_heads, spec.head_dim), spec.torch_dtype,
                 value_seed(spec, layer, 7), device)
    vn = _normal((num_tokens, spec.num_kv_heads, spec.head_dim), spec.torch_dtype,
                 value_seed(spec, layer, 8), device)
    return q, kn, vn


def new_token_counts(context_lens, seed: int, max_chunk: int, decode_frac: float = 0.5) -> np.ndarray:
    """New tokens per sequence in a mixed step: a seeded share of decodes (1
    token), the others a chunk of 2 .. min(context, max_chunk) tokens (a
    whole prompt when the chunk reaches the context)."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    n = np.ones(len(ctx), dtype=np.int32)
    for s, c in enumerate(ctx):
        if c >= 2 and rng.random() >= decode_frac:
            n[s] = int(rng.integers(2, min(int(c), max_chunk) + 1))
    return n


def small_spec(name="custom", *, num_q_heads=4, num_kv_heads=2, head_dim=64,
               block_size=16, dtype="f32", seed=11, ctx=(1, 15, 16, 17, 33),
               num_blocks=0, scale=0.0, kv_dtype="", kv_scales=(1.0, 1.0)) -> WorkloadSpec:
    """A small spec with explicit lengths, for edge-case tests."""
    ctx = tuple(int(c) for c in ctx)
    need = sum((c + block_size - 1) // block_size for c in ctx)
    return WorkloadSpec(name=name, num_layers=1, num_seqs=len(ctx), num_q_heads=num_q_heads,
                        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                        dtype=dtype, seed=seed, ctx_dist="list", ctx_list=ctx,
                        num_blocks=num_blocks or max(1, 2 * need), scale=scale,
                        kv_dtype=kv_dtype, kv_scales=tuple(kv_scales))


def prefix_request_trace(seed: int, num_ops: int, *, num_prompts: int = 6, vocab: int = 50,
                         max_shared: int = 40, max_own: int = 24, free_prob: float = 0.45):
    """A seeded stream of request arrivals and departures for a prefix-caching
    block pool: ("allocate", tokens) and ("free", index of an earlier live
    allocation, counted in arrival order).  Requests draw one of `num_prompts`
    shared prompts (some of it, all of it, or none) and append their own
    random tokens, so hits, partial hits, exact repeats and misses all occur.
    Token ids are small so that equal blocks in unrelated positions occur too.
    """
    rng = np.random.default_rng(seed)
    prompts = [rng.integers(0, vocab, size=max_shared).tolist() for _ in range(num_prompts)]
    ops = []
    live = 0
    for _ in range(num_ops):
        if live and rng.random() < free_prob:
            ops.append(("free", int(rng.integers(0, live))))
            live -= 1
            continue
        p = prompts[int(rng.integers(0, num_prompts))]
        shared = int(rng.choice([0, int(rng.integers(1, max_shared + 1)), max_shared]))
        own = int(rng.integers(0, max_own + 1))
        tokens = p[:shared] + rng.integers(0, vocab, size=own).tolist()
        if not tokens:
            tokens = [int(rng.integers(0, vocab))]
        ops.append(("allocate", tokens))
        live += 1
    return ops
