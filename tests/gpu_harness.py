"""Helpers of the GPU parity tests.

Inputs come from `workloads` only.  The CUDA side runs through the library's
C ABI (via the Python binding); the expected values come from `oracle` only,
computed on the host from the same inputs (the pre-append pool, the new rows,
the tables).  Nothing computed by the CUDA path is fed to the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_slots_gb300 as pkv
from workloads import fill_pool_layer, pool_layer_values, step_layer_values

# max |out - oracle| for fp32 output (fp16/bf16 inputs, fp32 accumulation).
ATOL = 2e-3


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int32) if t.element_size() == 4 else t.view(torch.int16)


def half_ulp(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Half a unit in the last place of `dtype` at |ref| (rounding of the final cast)."""
    if dtype == torch.float32:
        return np.abs(ref) * 2.0 ** -24
    mant = 10 if dtype == torch.float16 else 7
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14)))
    return 2.0 ** (e - mant - 1)


def check_output(out: torch.Tensor, ref: np.ndarray, what: str):
    got = out.detach().float().cpu().double().numpy()
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + (0 if out.dtype == torch.float32 else half_ulp(ref, out.dtype))
    worst = float(np.max(err - bound)) if err.size else -1.0
    assert worst <= 0, f"{what}: max |err| {float(err.max()):.3e} exceeds bound by {worst:.3e}"
    return float(err.max()) if err.size else 0.0


def ordered_bits(t: torch.Tensor) -> torch.Tensor:
    """Bit patterns of a 16- or 32-bit float tensor mapped to integers that
    increase with the value (so that two values' distance in ulps is the
    difference of their images); -0 and +0 map to 0."""
    b = bits(t).to(torch.int64)
    width = 8 * t.element_size()
    mag = b & ((1 << (width - 1)) - 1)
    return torch.where(b < 0, -mag, mag)


def check_cast(outq: torch.Tensor, out32: torch.Tensor, what: str, max_ulps: int = 1):
    """The fp16/bf16 output is the fp32 output of the same computation rounded
    to nearest even into that type, within `max_ulps` units in the last place
    (the final fold of a separate call may round one fp32 ulp differently)."""
    assert outq.dtype in (torch.float16, torch.bfloat16) and out32.dtype == torch.float32
    ref = out32.to(outq.dtype)  # round to nearest even
    d = (ordered_bits(outq.contiguous()) - ordered_bits(ref.contiguous())).abs()
    worst = int(d.max().item()) if d.numel() else 0
    assert worst <= max_ulps, f"{what}: {outq.dtype} output {worst} ulps from the rounded fp32 output"
    return worst


def _ws_opts(opts):
    return {k: v for k, v in opts.items() if k not in ("test_stall", "k_scale", "v_scale")}


def attend(q, kc, vc, tables, ctx, scale, out_dtype=None, **opts):
    """paged_decode_attention with a NaN-filled output and an 0xFF-filled
    workspace, so that an output the kernels fail to write, or a partial they
    read without having written it, cannot pass unnoticed.  An E4M3 cache
    takes k_scale and v_scale in opts."""
    B, Hq, D = q.shape
    out_dtype = out_dtype or q.dtype
    out = torch.full((B, Hq, D), float("nan"), dtype=out_dtype, device=q.device)
    n = pkv.workspace_bytes(B, Hq, kc.shape[1], D, q.device, **_ws_opts(opts))
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=q.device)
    pkv.workspace_init(ws, B, kc.shape[1])  # only the merge counters must start at zero
    return pkv.paged_decode_attention(q, kc, vc, tables, ctx, scale, out=out, out_dtype=out_dtype,
                                      workspace=ws, **opts)


def attend_append(q, kn, vn, kc, vc, tables, ctx, scale, seq_ids=None, out_dtype=None, **opts):
    """paged_decode_append_attention with poisoned output/workspace; returns (out, slots)."""
    B, Hq, D = q.shape
    out_dtype = out_dtype or q.dtype
    out = torch.full((B, Hq, D), float("nan"), dtype=out_dtype, device=q.device)
    slots = torch.full((B,), -7, dtype=torch.int32, device=q.device)
    n = pkv.workspace_bytes(B, Hq, kc.shape[1], D, q.device, **_ws_opts(opts))
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=q.device)
    pkv.workspace_init(ws, B, kc.shape[1])
    pkv.paged_decode_append_attention(q, kn, vn, kc, vc, tables, ctx, scale, seq_ids=seq_ids, out=out,
                                      out_dtype=out_dtype, slot_mapping=slots, workspace=ws, **opts)
    return out, slots


def scale_opts(spec) -> dict:
    """k_scale / v_scale arguments of an E4M3 spec (none otherwise)."""
    return dict(k_scale=spec.kv_scales[0], v_scale=spec.kv_scales[1]) if spec.fp8 else {}


def oracle_append(spec, k_pre, v_pre, kn, vn, slots):
    """The oracle's append for the spec's cache type."""
    if spec.fp8:
        return oracle.append_e4m3(k_pre, v_pre, kn, vn, slots, *spec.kv_scales)
    return oracle.append(k_pre, v_pre, kn, vn, slots)


def oracle_attention(spec, q, k, v, tables, ctx):
    return oracle.paged_decode(q, k, v, tables, ctx, spec.attn_scale, **scale_opts(spec))


def take(t: torch.Tensor, idx: torch.Tensor) -> torch.Tensor:
    """t[idx] along dim 0 (through a byte view for one-byte types)."""
    if t.element_size() == 1:
        return t.view(torch.uint8)[idx].view(t.dtype)
    return t[idx]


def cache_bits(t: torch.Tensor) -> torch.Tensor:
    """Bit patterns of a cache of any type (E4M3 as bytes)."""
    return t.view(torch.uint8) if t.element_size() == 1 else bits(t)


def newest_slot_masks(placement):
    """seq_ids passed to the append: -1 marks a sequence that writes nothing."""
    return np.where(placement.appends, np.arange(len(placement.appends)), -1).astype(np.int32)


class SmallCase:
    """A workload small enough that the oracle checks every output; host copies kept."""

    def __init__(self, spec, placement, layer=0):
        self.spec, self.pl, self.layer = spec, placement, layer
        self.kpool, self.vpool = pool_layer_values(spec, placement.num_blocks, layer, "cpu")
        self.q, self.kn, self.vn = step_layer_values(spec, len(placement.context_lens), layer, "cpu")

    def oracle(self):
        """(slots, K after append, V after append, fp64 attention output)."""
        sl = oracle.slot_mapping(self.pl.block_tables, self.pl.context_lens, self.spec.block_size)
        sl_w = np.where(self.pl.appends, sl, -1).astype(np.int32)
        kpost, vpost = oracle_append(self.spec, self.kpool, self.vpool, self.kn, self.vn, sl_w)
        ref = oracle_attention(self.spec, self.q, kpost, vpost, self.pl.block_tables,
                               self.pl.context_lens)
        return sl, kpost, vpost, ref

    def device(self, dev="cuda"):
        s = self.spec
        pool = pkv.KVPool(s.num_layers, self.pl.num_blocks, s.block_size, s.num_kv_heads,
                          s.head_dim, s.cache_torch_dtype, device=dev)
        kc, vc = pool.layer(self.layer)
        kc.copy_(self.kpool)
        vc.copy_(self.vpool)
        d = dict(pool=pool, kc=kc, vc=vc,
                 tables=torch.from_numpy(self.pl.block_tables).to(dev),
                 ctx=torch.from_numpy(self.pl.context_lens).to(dev),
                 seq_ids=torch.from_numpy(newest_slot_masks(self.pl)).to(dev),
                 q=self.q.to(dev), kn=self.kn.to(dev), vn=self.vn.to(dev))
        return d


def run_step(d, spec, num_blocks, layer=0, out_dtype=None, **opts):
    """Slot mapping, append and attention of one layer through the library."""
    slots = pkv.slot_mapping(d["tables"], d["ctx"], spec.block_size, num_blocks)
    d["pool"].append(layer, d["kn"], d["vn"], slots, seq_ids=d["seq_ids"], **scale_opts(spec))
    out = attend(d["q"], d["kc"], d["vc"], d["tables"], d["ctx"], spec.attn_scale,
                 out_dtype=out_dtype, **scale_opts(spec), **opts)
    return slots, out


def compact_blocks(tables: np.ndarray, seqs) -> tuple[np.ndarray, np.ndarray]:
    """Physical blocks used by `seqs` and their tables renumbered into that list."""
    rows = tables[seqs]
    used = np.unique(rows[rows >= 0])
    remap = np.full(int(tables.max()) + 1, -1, dtype=np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    new = np.where(rows >= 0, remap[np.maximum(rows, 0)], -1).astype(np.int32)
    return used, new


class LargeCase:
    """A full-size workload generated on the device; the oracle checks sampled sequences."""

    def __init__(self, spec, placement, dev="cuda"):
        self.spec, self.pl, self.dev = spec, placement, dev
        s = spec
        self.pool = pkv.KVPool(s.num_layers, placement.num_blocks, s.block_size, s.num_kv_heads,
                               s.head_dim, s.cache_torch_dtype, device=dev)
        self.tables = torch.from_numpy(placement.block_tables).to(dev)
        self.ctx = torch.from_numpy(placement.context_lens).to(dev)
        self.seq_ids = torch.from_numpy(newest_slot_masks(placement)).to(dev)

    def fill(self, layer):
        kc, vc = self.pool.layer(layer)
        fill_pool_layer(self.spec, layer, kc, vc)
        q, kn, vn = step_layer_values(self.spec, len(self.pl.context_lens), layer, self.dev)
        return kc, vc, q, kn, vn

    def check_layer(self, layer, seqs=None, fused=False, whole_pool=True, **opts):
        """Run one layer on the full batch; compare with the oracle.

        seqs: the sequences whose outputs are checked (None: every sequence).
        whole_pool: bit-compare the whole layer pool after the append with the
        oracle's scatter of every sequence's new rows into a host copy of the
        pre-step pool (else only the blocks of `seqs`, over a compact copy).
        fused: append and attention in one call (paged_decode_append_attention).
        Returns (max err of the fp32 output, of the q-dtype output, fp32 output
        on the device, q-dtype output on the device)."""
        s, pl = self.spec, self.pl
        B = len(pl.context_lens)
        seqs = np.arange(B) if seqs is None else np.asarray(seqs, dtype=np.int64)
        kc, vc, q, kn, vn = self.fill(layer)
        if whole_pool:
            k_pre, v_pre = kc.cpu(), vc.cpu()  # the oracle's pool: pre-append, every block
        else:
            used, ctab = compact_blocks(pl.block_tables, seqs)
            used_t = torch.from_numpy(used.astype(np.int64)).to(self.dev)
            k_pre, v_pre = take(kc, used_t).cpu(), take(vc, used_t).cpu()
        so = scale_opts(s)
        if fused:
            out32, slots = attend_append(q, kn, vn, kc, vc, self.tables, self.ctx, s.attn_scale,
                                         seq_ids=self.seq_ids, out_dtype=torch.float32, **so, **opts)
        else:
            slots = pkv.slot_mapping(self.tables, self.ctx, s.block_size, pl.num_blocks)
            self.pool.append(layer, kn, vn, slots, seq_ids=self.seq_ids, **so)
            out32 = attend(q, kc, vc, self.tables, self.ctx, s.attn_scale, out_dtype=torch.float32,
                           **so, **opts)
        outq = attend(q, kc, vc, self.tables, self.ctx, s.attn_scale, **so, **opts)
        st, flags = pkv.device_status()
        assert st == 0 and flags == 0, f"device status {st} flags {flags:#x}"
        ctx_s = pl.context_lens[seqs]
        o_full = oracle.slot_mapping(pl.block_tables, pl.context_lens, s.block_size)
        # Device slot mapping: bit-exact for every sequence (real table).
        assert np.array_equal(slots.cpu().numpy(), o_full), "slot mapping"
        if whole_pool:
            o_sl = np.where(pl.appends, o_full, -1).astype(np.int32)
            k_post, v_post = oracle_append(s, k_pre, v_pre, kn.cpu(), vn.cpu(), o_sl)
            assert torch.equal(cache_bits(kc.cpu()), cache_bits(k_post)), "K pool after append"
            assert torch.equal(cache_bits(vc.cpu()), cache_bits(v_post)), "V pool after append"
            tab = pl.block_tables[seqs]
        else:
            o_sl = oracle.slot_mapping(ctab, ctx_s, s.block_size)
            o_sl = np.where(pl.appends[seqs], o_sl, -1).astype(np.int32)
            k_post, v_post = oracle_append(s, k_pre, v_pre, kn[seqs].cpu(), vn[seqs].cpu(), o_sl)
            assert torch.equal(cache_bits(take(kc, used_t).cpu()), cache_bits(k_post)), "K blocks after append"
            assert torch.equal(cache_bits(take(vc, used_t).cpu()), cache_bits(v_post)), "V blocks after append"
            tab = ctab
        ref = oracle_attention(s, q[seqs].cpu(), k_post, v_post, tab, ctx_s)
        del k_pre, v_pre, k_post, v_post
        idx = torch.as_tensor(seqs, device=self.dev)
        e32 = check_output(out32[idx], ref, f"{s.name} layer {layer} fp32 out")
        eq = check_output(outq[idx], ref, f"{s.name} layer {layer} {s.dtype} out")
        check_cast(outq, out32, f"{s.name} layer {layer}")
        return e32, eq, out32, outq

    def solo_agreement(self, layer, seqs, batch_out32, **opts):
        """Each sequence of `seqs` attended alone (a batch of one: its table
        row and length, the same pool) against its row of the full batch's
        fp32 output.  Returns (max |difference|, sequences whose bits agree)."""
        s = self.spec
        kc, vc = self.pool.layer(layer)
        q, _, _ = step_layer_values(s, len(self.pl.context_lens), layer, self.dev)
        worst, same = 0.0, 0
        for i in seqs:
            i = int(i)
            one = attend(q[i:i + 1].contiguous(), kc, vc, self.tables[i:i + 1].contiguous(),
                         self.ctx[i:i + 1].contiguous(), s.attn_scale, out_dtype=torch.float32,
                         **scale_opts(s), **opts)
            d = (one[0] - batch_out32[i]).abs().max().item()
            worst = max(worst, d)
            same += int(torch.equal(bits(one[0]), bits(batch_out32[i])))
        assert pkv.device_status() == (0, 0)
        return worst, same


def sample_sequences(placement, n, seed):
    """n sequences: the longest, the shortest, and a seeded draw of the rest."""
    ctx = placement.context_lens
    order = np.argsort(ctx, kind="stable")
    pick = {int(order[0]), int(order[-1])}
    rng = np.random.default_rng(seed)
    rest = [i for i in range(len(ctx)) if i not in pick]
    pick.update(int(x) for x in rng.choice(rest, size=min(n - len(pick), len(rest)), replace=False))
    return np.array(sorted(pick), dtype=np.int64)
