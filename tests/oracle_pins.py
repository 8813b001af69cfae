"""Checks that tie the oracle to facts other than itself.

Each check takes a loaded oracle library and raises AssertionError on a
mismatch.  test_oracle_pins.py runs them against the real oracle, and runs
them again against copies of the oracle with one deliberate mistake each, to
show that every plausible mistake is caught by at least one check.

What pins what:
  decoders     -- numpy's binary16 and torch's bfloat16 conversions, all 65536
                  bit patterns.
  slots        -- the worked slots printed in "vLLM Architecture and
                  Installation", Example 3 (A token 9 -> 13, A token 12 -> 24,
                  B token 7 -> 23).
  append       -- scatter then block-level read-back gives the contiguous draw
                  back, untouched slots keep their sentinel, slot -1 is skipped.
  attention    -- brute force over unpaged per-sequence arrays (pool assembled
                  block by block with numpy slicing, softmax from scipy),
                  closed forms (equal keys or zero scale give the mean of V,
                  one token gives that token's V, a two-token case by hand),
                  an overwhelming score (exercises the max subtraction),
                  physical-block relabelling, equal heads in a group.
  e4m3         -- torch's float8_e4m3fn conversions: decode of all 256 codes,
                  encode of every midpoint between neighbouring codes (ties to
                  even) and of random values below the overflow threshold;
                  round trip of every finite code; the format's landmarks
                  (1.0, 448, 2^-6, 2^-9); saturation from 448 up (the
                  satfinite reading; torch itself gives NaN there).
  fp8 append   -- the quantizing scatter reads back as torch's cast of the
                  fp32 quotient x / scale; untouched slots keep their codes.
  fp8 attention-- equals the brute force over the dequantized cache
                  (scale * value), with different K and V scales.
  multi-token  -- torch's causal scaled_dot_product_attention for whole
                  prompts; a brute force over the causal prefix after earlier
                  context; chunking a prompt changes no row; one new token is
                  the decode step; the worked slots of Example 3 for new
                  tokens at several positions.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- decoders
def check_f16_decoder(lib):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_values(bits, "f16", lib=lib)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(got, ref, equal_nan=True), "binary16 decoder"


def check_bf16_decoder(lib):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_values(bits, "bf16", lib=lib)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, ref, equal_nan=True), "bfloat16 decoder"


def check_f32_decoder(lib):
    x = np.random.default_rng(5).standard_normal(4096).astype(np.float32)
    x[:4] = [0.0, -0.0, 1e-42, 3.4e38]
    got = oracle.decode_values(x, "f32", lib=lib)
    assert np.array_equal(got, x.astype(np.float64)), "binary32 decoder"


# -------------------------------------------------------------------- slots
def check_worked_slots(lib):
    g = golden("block_tables_vllm_example3.json")
    bs = g["block_size"]
    check = [s for s in g["steps"] if s.get("label") == "after 3 decode steps"][0]
    names = sorted(check["tables"])
    width = max(len(t) for t in check["tables"].values())
    tables = np.full((len(names), width), -1, dtype=np.int32)
    for i, n in enumerate(names):
        tables[i, :len(check["tables"][n])] = check["tables"][n]
    expect = [s for s in g["steps"] if s["op"] == "slots"][0]["expect"]
    for name, pos, slot in expect:
        got = oracle.slot(tables, names.index(name), pos, bs, lib=lib)
        assert got == slot, f"slot of {name} token {pos}: {got} != {slot}"
    # Newest-token slots of a step in which A has 13 and B has 8 tokens.
    lens = np.array([check["lengths"][n] for n in names], dtype=np.int32)
    got = oracle.slot_mapping(tables, lens, bs, lib=lib)
    assert got.tolist() == [24, 23], got
    assert oracle.slot_mapping(tables, np.array([0, 0], np.int32), bs, lib=lib).tolist() == [-1, -1]


# ------------------------------------------------------------------- append
def _random_tables(rng, ctx, bs, NB):
    nblk = [(c + bs - 1) // bs for c in ctx]
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((len(ctx), max(1, max(nblk))), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[cur:cur + n]
        cur += n
    return tables


def check_append_roundtrip(lib):
    rng = np.random.default_rng(21)
    for dtype, np_dt in (("f32", np.float32), ("f16", np.float16)):
        bs, Hkv, D, NB = 4, 3, 8, 24
        ctx = [5, 1, 9, 4]
        tables = _random_tables(rng, ctx, bs, NB)
        sentinel = np.full((NB, Hkv, bs, D), -7.0, dtype=np_dt)
        Kc = [rng.standard_normal((Hkv, c, D)).astype(np_dt) for c in ctx]
        Vc = [rng.standard_normal((Hkv, c, D)).astype(np_dt) for c in ctx]
        kp, vp = torch.from_numpy(sentinel.copy()), torch.from_numpy(sentinel.copy())
        # Append position by position, as decode steps would, one call per step.
        for pos in range(max(ctx)):
            rows = [s for s, c in enumerate(ctx) if pos < c]
            slots = np.array([oracle.slot(tables, s, pos, bs, lib=lib) for s in rows], np.int32)
            slots = np.concatenate([slots, np.array([-1], np.int32)])  # a padding token
            kn = np.stack([Kc[s][:, pos] for s in rows] + [np.full((Hkv, D), 99, np_dt)])
            vn = np.stack([Vc[s][:, pos] for s in rows] + [np.full((Hkv, D), 99, np_dt)])
            kp, vp = oracle.append(kp, vp, torch.from_numpy(kn), torch.from_numpy(vn), slots, lib=lib)
        kp, vp = kp.numpy(), vp.numpy()
        touched = np.zeros((NB, bs), dtype=bool)
        for s, c in enumerate(ctx):
            for j in range((c + bs - 1) // bs):
                m = min(bs, c - j * bs)
                blk = tables[s, j]
                assert np.array_equal(kp[blk, :, :m, :], Kc[s][:, j * bs:j * bs + m, :]), "K read-back"
                assert np.array_equal(vp[blk, :, :m, :], Vc[s][:, j * bs:j * bs + m, :]), "V read-back"
                touched[blk, :m] = True
        untouched = ~touched
        assert np.all(kp.transpose(0, 2, 1, 3)[untouched] == np_dt(-7.0)), "K slot written that should not be"
        assert np.all(vp.transpose(0, 2, 1, 3)[untouched] == np_dt(-7.0)), "V slot written that should not be"
    # A slot past the end of the pool is an error.
    try:
        oracle.append(torch.zeros(2, 1, 4, 8), torch.zeros(2, 1, 4, 8), torch.zeros(1, 1, 8),
                      torch.zeros(1, 1, 8), np.array([8], np.int32), lib=lib)
    except ValueError:
        pass
    else:
        raise AssertionError("append accepted a slot outside the pool")


# ---------------------------------------------------------------- attention
def assemble_pool(Kc, Vc, tables, NB, bs, fill_rng, np_dt):
    """Pool built block by block from per-sequence arrays [Hkv, ctx, D].

    Unused slots hold random values, so a gather that strays reads garbage."""
    Hkv, _, D = Kc[0].shape
    kp = fill_rng.standard_normal((NB, Hkv, bs, D)).astype(np_dt)
    vp = fill_rng.standard_normal((NB, Hkv, bs, D)).astype(np_dt)
    for s in range(len(Kc)):
        c = Kc[s].shape[1]
        for j in range((c + bs - 1) // bs):
            m = min(bs, c - j * bs)
            kp[tables[s, j], :, :m, :] = Kc[s][:, j * bs:j * bs + m, :]
            vp[tables[s, j], :, :m, :] = Vc[s][:, j * bs:j * bs + m, :]
    return kp, vp


def dense_attention(q, Kc, Vc, scale, G):
    """Unpaged softmax attention with scipy's softmax, fp64."""
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D))
    for s in range(B):
        if Kc[s].shape[1] == 0:
            continue
        for g in range(Hq):
            k = Kc[s][g // G].astype(np.float64)
            v = Vc[s][g // G].astype(np.float64)
            w = scipy.special.softmax(scale * (k @ q[s, g].astype(np.float64)))
            out[s, g] = w @ v
    return out


def _case(rng, ctx, Hq, Hkv, D, bs, np_dt, spare=5):
    NB = sum((c + bs - 1) // bs for c in ctx) + spare
    tables = _random_tables(rng, ctx, bs, NB)
    Kc = [rng.standard_normal((Hkv, c, D)).astype(np_dt) for c in ctx]
    Vc = [rng.standard_normal((Hkv, c, D)).astype(np_dt) for c in ctx]
    q = rng.standard_normal((len(ctx), Hq, D)).astype(np_dt)
    kp, vp = assemble_pool(Kc, Vc, tables, NB, bs, rng, np_dt)
    return q, Kc, Vc, tables, kp, vp


def _run(lib, q, kp, vp, tables, ctx, scale, threads=0):
    return oracle.paged_decode(torch.from_numpy(q), torch.from_numpy(kp), torch.from_numpy(vp),
                               tables, np.array(ctx, np.int32), scale, nthreads=threads, lib=lib)


def check_bruteforce(lib):
    rng = np.random.default_rng(33)
    cases = [
        # ctx, Hq, Hkv, D, bs
        ([1, 3, 4, 5, 8, 9], 4, 2, 8, 4),
        ([17, 64, 100, 31], 8, 2, 16, 16),
        ([7, 0, 12], 3, 3, 8, 4),      # G = 1 (multi-head attention), an empty sequence
        ([33, 2], 8, 1, 8, 8),         # all heads share one KV head
        ([15, 16, 17, 32], 8, 4, 32, 16),
    ]
    for ctx, Hq, Hkv, D, bs in cases:
        for np_dt in (np.float32, np.float16):
            q, Kc, Vc, tables, kp, vp = _case(rng, ctx, Hq, Hkv, D, bs, np_dt)
            scale = 1.0 / math.sqrt(D)
            got = _run(lib, q, kp, vp, tables, ctx, scale)
            ref = dense_attention(q, Kc, Vc, scale, Hq // Hkv)
            err = np.max(np.abs(got - ref)) if got.size else 0.0
            assert err < 1e-12, f"brute force {ctx} {np_dt.__name__}: {err}"


def check_closed_forms(lib):
    rng = np.random.default_rng(44)
    bs, Hkv, Hq, D = 4, 2, 4, 8
    ctx = [6, 1, 11]
    q, Kc, Vc, tables, kp, vp = _case(rng, ctx, Hq, Hkv, D, bs, np.float32)
    # Equal keys: every token gets the same weight -> mean of V.
    Ke = [np.repeat(k[:, :1, :], k.shape[1], axis=1) for k in Kc]
    kp2, vp2 = assemble_pool(Ke, Vc, tables, kp.shape[0], bs, rng, np.float32)
    got = _run(lib, q, kp2, vp2, tables, ctx, 0.7)
    for s in range(len(ctx)):
        for g in range(Hq):
            mean = Vc[s][g // 2].astype(np.float64).mean(axis=0)
            assert np.max(np.abs(got[s, g] - mean)) < 1e-12, "equal keys -> mean of V"
    # Zero scale: mean of V as well.
    got = _run(lib, q, kp, vp, tables, ctx, 0.0)
    for s in range(len(ctx)):
        for g in range(Hq):
            mean = Vc[s][g // 2].astype(np.float64).mean(axis=0)
            assert np.max(np.abs(got[s, g] - mean)) < 1e-12, "scale 0 -> mean of V"
    # One token: that token's V, exactly.
    got = _run(lib, q, kp, vp, tables, ctx, 0.3)
    for g in range(Hq):
        assert np.array_equal(got[1, g], Vc[1][g // 2][0].astype(np.float64)), "one token -> its V"
    # Two tokens by hand: q = a e0, k0 = e0, k1 = 0 -> weights e^(s a)/(e^(s a)+1), 1/(e^(s a)+1).
    a, sc = 2.0, 0.5
    q2 = np.zeros((1, 1, D), np.float32)
    q2[0, 0, 0] = a
    K2 = [np.zeros((1, 2, D), np.float32)]
    K2[0][0, 0, 0] = 1.0
    V2 = [np.zeros((1, 2, D), np.float32)]
    V2[0][0, 0, :] = 3.0
    V2[0][0, 1, :] = -1.0
    t2 = np.array([[1]], np.int32)
    kp3, vp3 = assemble_pool(K2, V2, t2, 3, 2, rng, np.float32)
    got = _run(lib, q2, kp3, vp3, t2, [2], sc)
    e = math.exp(sc * a)
    want = (3.0 * e - 1.0) / (e + 1.0)
    assert np.max(np.abs(got[0, 0] - want)) < 1e-14, "two-token closed form"
    # An overwhelming score (exp would overflow without the max subtraction):
    # the output is the V of the winning token.
    q4 = np.zeros((1, 1, D), np.float32)
    q4[0, 0, :] = 1.0
    K4 = [np.zeros((1, 3, D), np.float32)]
    K4[0][0, 1, :] = 2000.0
    K4[0][0, 0, :] = 1000.0
    V4 = [rng.standard_normal((1, 3, D)).astype(np.float32)]
    t4 = np.array([[2]], np.int32)
    kp4, vp4 = assemble_pool(K4, V4, t4, 3, 4, rng, np.float32)
    got = _run(lib, q4, kp4, vp4, t4, [3], 1.0)
    assert np.all(np.isfinite(got)), "overflow in softmax"
    assert np.array_equal(got[0, 0], V4[0][0, 1].astype(np.float64)), "winner's V"


def check_relabel_and_heads(lib):
    rng = np.random.default_rng(55)
    bs, Hkv, Hq, D = 4, 2, 6, 8
    ctx = [9, 4, 13, 1]
    q, Kc, Vc, tables, kp, vp = _case(rng, ctx, Hq, Hkv, D, bs, np.float16)
    base = _run(lib, q, kp, vp, tables, ctx, 0.35)
    # Relabel physical blocks: pool'[pi[b]] = pool[b], table' = pi[table].
    NB = kp.shape[0]
    pi = rng.permutation(NB).astype(np.int32)
    kq, vq = np.empty_like(kp), np.empty_like(vp)
    kq[pi], vq[pi] = kp, vp
    t2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1).astype(np.int32)
    assert np.array_equal(_run(lib, q, kq, vq, t2, ctx, 0.35), base), "relabelled blocks"
    # Equal query heads within a group give equal outputs.
    qe = q.copy()
    qe[:, 1] = qe[:, 0]
    qe[:, 2] = qe[:, 0]
    got = _run(lib, qe, kp, vp, tables, ctx, 0.35)
    assert np.array_equal(got[:, 1], got[:, 0]) and np.array_equal(got[:, 2], got[:, 0]), "equal heads"
    # Thread count does not change the result.
    assert np.array_equal(_run(lib, q, kp, vp, tables, ctx, 0.35, threads=1), base), "threads"
    # Two sequences sharing a table and q give equal outputs.
    t3 = tables.copy()
    t3[1] = t3[0]
    q3 = q.copy()
    q3[1] = q3[0]
    c3 = list(ctx)
    c3[1] = c3[0]
    got = _run(lib, q3, kp, vp, t3, c3, 0.35)
    assert np.array_equal(got[1], got[0]), "shared table"


# --------------------------------------------------------------------- E4M3
def _torch_e4m3_codes(x_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def check_e4m3_decoder(lib):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_values(codes, "e4m3", lib=lib)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(got, ref, equal_nan=True), "E4M3 decoder"
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]), "E4M3 NaN codes"
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x08] == 2.0**-6 and got[0x01] == 2.0**-9


def check_e4m3_encoder(lib):
    enc = lambda x: oracle.e4m3_encode(x, lib=lib)  # noqa: E731
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.decode_values(codes, "e4m3", lib=lib)
    for c, v in zip(codes, vals):
        assert enc(float(v)) == c, f"round trip of code {c:#x}"
    # Midpoints between neighbouring non-negative codes: exact ties.
    pos = np.sort(vals[vals >= 0])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal((pos[:-1] + pos[1:]) / 2, mids.astype(np.float64)), "midpoints exact in fp32"
    got = np.array([enc(float(m)) for m in mids], dtype=np.uint8)
    assert np.array_equal(got, _torch_e4m3_codes(mids)), "ties to even"
    got = np.array([enc(float(-m)) for m in mids], dtype=np.uint8)
    assert np.array_equal(got, _torch_e4m3_codes(-mids)), "negative ties"
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.uniform(-463.9, 463.9, 3000), rng.standard_normal(3000) * 2.0**-7,
                        rng.standard_normal(1000)]).astype(np.float32)
    got = np.array([enc(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, _torch_e4m3_codes(x)), "random values"
    for v in (448.0, 463.99, 464.0, 1e6, float("inf")):
        assert enc(v) == 0x7E and enc(-v) == 0xFE, f"saturation at {v}"
    assert enc(float("nan")) == 0x7F
    assert enc(-0.0) == 0x80 and enc(0.0) == 0x00


def check_fp8_append(lib):
    rng = np.random.default_rng(31)
    bs, Hkv, D, NB, n = 4, 2, 8, 6, 5
    sentinel = np.full((NB, Hkv, bs, D), 0x55, np.uint8)
    kp = torch.from_numpy(sentinel.copy()).view(torch.float8_e4m3fn)
    vp = torch.from_numpy(sentinel.copy()).view(torch.float8_e4m3fn)
    kn = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    vn = torch.from_numpy(rng.standard_normal((n, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    slots = np.array([3, 22, -1, 9, 0], np.int32)
    ks, vs = 1.0 / 48.0, 0.0125
    K, V = oracle.append_e4m3(kp, vp, kn, vn, slots, ks, vs, lib=lib)
    K, V = K.view(torch.uint8).numpy(), V.view(torch.uint8).numpy()
    written = np.zeros((NB, bs), bool)
    for i, sl in enumerate(slots):
        if sl < 0:
            continue
        b, o = sl // bs, sl % bs
        kq = (kn[i].float() / torch.tensor(ks, dtype=torch.float32)).numpy()
        vq = (vn[i].float() / torch.tensor(vs, dtype=torch.float32)).numpy()
        assert np.array_equal(K[b, :, o, :], _torch_e4m3_codes(kq)), "K codes"
        assert np.array_equal(V[b, :, o, :], _torch_e4m3_codes(vq)), "V codes"
        written[b, o] = True
    assert np.all(K.transpose(0, 2, 1, 3)[~written] == 0x55) and np.all(V.transpose(0, 2, 1, 3)[~written] == 0x55)


def check_fp8_attention(lib):
    rng = np.random.default_rng(34)
    ctx, Hq, Hkv, D, bs = [5, 1, 19, 16], 8, 2, 16, 4
    NB = sum((c + bs - 1) // bs for c in ctx) + 3
    tables = _random_tables(rng, ctx, bs, NB)
    kp = torch.from_numpy(rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8))
    vp = torch.from_numpy(rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8))
    kp[(kp & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    vp[(vp & 0x7F) == 0x7F] = 0x44
    q = torch.from_numpy(rng.standard_normal((len(ctx), Hq, D)).astype(np.float32)).to(torch.bfloat16)
    ks, vs, scale = 0.004, 0.07, 0.25
    got = oracle.paged_decode(q, kp.view(torch.float8_e4m3fn), vp.view(torch.float8_e4m3fn), tables,
                              np.array(ctx, np.int32), scale, lib=lib, k_scale=ks, v_scale=vs)
    kf = ks * kp.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vf = vs * vp.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    Kc = [np.concatenate([kf[tables[s, j]] for j in range((c + bs - 1) // bs)], axis=1)[:, :c] for s, c in enumerate(ctx)]
    Vc = [np.concatenate([vf[tables[s, j]] for j in range((c + bs - 1) // bs)], axis=1)[:, :c] for s, c in enumerate(ctx)]
    ref = dense_attention(q.to(torch.float64).numpy(), Kc, Vc, scale, Hq // Hkv)
    assert np.max(np.abs(got - ref)) < 1e-12, "fp8 attention vs dequantized brute force"


# ------------------------------------------------------ multi-token queries
def _prefill_case(rng, ctx, nq, Hq, Hkv, D, bs, np_dt):
    """Paged pool plus dense per-sequence arrays for a multi-token step."""
    q_, Kc, Vc, tables, kp, vp = _case(rng, ctx, Hq, Hkv, D, bs, np_dt)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = rng.standard_normal((int(qs[-1]), Hq, D)).astype(np_dt)
    return q, qs, Kc, Vc, tables, kp, vp


def _run_prefill(lib, q, kp, vp, tables, qs, ctx, scale, threads=0):
    return oracle.paged_prefill(torch.from_numpy(q), torch.from_numpy(kp), torch.from_numpy(vp), tables, qs,
                                np.array(ctx, np.int32), scale, nthreads=threads, lib=lib)


def check_prefill_vs_torch_sdpa(lib):
    # Whole prompts (no earlier context): causal attention, which torch's
    # scaled_dot_product_attention computes directly (fp64, heads expanded).
    rng = np.random.default_rng(61)
    ctx = [1, 7, 16, 23]
    Hq, Hkv, D, bs = 6, 2, 16, 4
    q, qs, Kc, Vc, tables, kp, vp = _prefill_case(rng, ctx, ctx, Hq, Hkv, D, bs, np.float32)
    scale = 0.3
    got = _run_prefill(lib, q, kp, vp, tables, qs, ctx, scale)
    for s, c in enumerate(ctx):
        qq = torch.from_numpy(q[qs[s]:qs[s + 1]].astype(np.float64)).permute(1, 0, 2)  # [Hq, n, D]
        kk = torch.from_numpy(Kc[s].astype(np.float64)).repeat_interleave(Hq // Hkv, dim=0)
        vv = torch.from_numpy(Vc[s].astype(np.float64)).repeat_interleave(Hq // Hkv, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=scale)
        err = np.max(np.abs(got[qs[s]:qs[s + 1]] - ref.permute(1, 0, 2).numpy()))
        assert err < 1e-12, f"causal SDPA, sequence {s}: {err}"


def check_prefill_bruteforce_with_context(lib):
    # Chunks after earlier context, mixed with single-token decodes.
    rng = np.random.default_rng(62)
    ctx = [9, 1, 40, 17, 5]
    nq = [4, 1, 13, 1, 5]
    Hq, Hkv, D, bs = 8, 2, 8, 4
    q, qs, Kc, Vc, tables, kp, vp = _prefill_case(rng, ctx, nq, Hq, Hkv, D, bs, np.float16)
    scale = 0.5
    got = _run_prefill(lib, q, kp, vp, tables, qs, ctx, scale)
    G = Hq // Hkv
    for s, (c, n) in enumerate(zip(ctx, nq)):
        for i in range(n):
            pos = c - n + i
            for g in range(Hq):
                k = Kc[s][g // G][:pos + 1].astype(np.float64)
                v = Vc[s][g // G][:pos + 1].astype(np.float64)
                w = scipy.special.softmax(scale * (k @ q[qs[s] + i, g].astype(np.float64)))
                assert np.max(np.abs(got[qs[s] + i, g] - w @ v)) < 1e-12, f"seq {s} token {i} head {g}"


def check_prefill_chunking_and_decode(lib):
    rng = np.random.default_rng(63)
    ctx = [21]
    Hq, Hkv, D, bs = 4, 2, 8, 4
    q, qs, Kc, Vc, tables, kp, vp = _prefill_case(rng, ctx, ctx, Hq, Hkv, D, bs, np.float32)
    whole = _run_prefill(lib, q, kp, vp, tables, qs, ctx, 0.4)
    # The same prompt in three chunks (8, 8, 5 tokens) gives the same rows.
    done = 0
    for n in (8, 8, 5):
        part = _run_prefill(lib, q[done:done + n], kp, vp, tables, np.array([0, n], np.int32), [done + n], 0.4)
        assert np.array_equal(part, whole[done:done + n]), "chunked = whole"
        done += n
    # A single new token is the decode step.
    dec = _run(lib, q[20:21], kp, vp, tables, [21], 0.4)
    assert np.array_equal(dec, whole[20:21]), "one new token = decode"


def check_fp8_prefill(lib):
    # Multi-token queries over an E4M3 cache with power-of-two scales: every
    # dequantized value (scale times the code's value) is exact in f32, so the
    # same step over an f32 cache holding those values must agree to rounding;
    # and one new token per sequence is the E4M3 decode step, bit for bit.
    rng = np.random.default_rng(65)
    ctx, nq = [9, 1, 30, 17], [4, 1, 11, 17]
    Hq, Hkv, D, bs = 8, 2, 16, 4
    NB = sum((c + bs - 1) // bs for c in ctx) + 3
    tables = _random_tables(rng, ctx, bs, NB)
    kp = torch.from_numpy(rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8))
    vp = torch.from_numpy(rng.integers(0, 256, (NB, Hkv, bs, D), dtype=np.uint8))
    kp[(kp & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    vp[(vp & 0x7F) == 0x7F] = 0x44
    k8, v8 = kp.view(torch.float8_e4m3fn), vp.view(torch.float8_e4m3fn)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    T = int(qs[-1])
    q = torch.from_numpy(rng.standard_normal((T, Hq, D)).astype(np.float32)).to(torch.bfloat16)
    ks, vs, scale = 2.0 ** -6, 2.0 ** -3, 0.3
    c = np.array(ctx, np.int32)
    got = oracle.paged_prefill(q, k8, v8, tables, qs, c, scale, lib=lib, k_scale=ks, v_scale=vs)
    kf = (ks * k8.to(torch.float64)).to(torch.float32)
    vf = (vs * v8.to(torch.float64)).to(torch.float32)
    ref = oracle.paged_prefill(q.float(), kf, vf, tables, qs, c, scale, lib=lib)
    assert np.max(np.abs(got - ref)) < 1e-12, "E4M3 prefill vs the f32 prefill over the dequantized cache"
    one = np.arange(len(ctx) + 1, dtype=np.int32)
    qd = q[qs[1:] - 1]  # each sequence's last new token
    dec = oracle.paged_decode(qd, k8, v8, tables, c, scale, lib=lib, k_scale=ks, v_scale=vs)
    pre = oracle.paged_prefill(qd, k8, v8, tables, one, c, scale, lib=lib, k_scale=ks, v_scale=vs)
    assert np.array_equal(pre, dec), "one new token over an E4M3 cache = the E4M3 decode step"
    assert np.array_equal(pre, got[qs[1:] - 1]), "the last token of each chunk"


def check_varlen_slots(lib):
    # The worked slots of "vLLM Architecture and Installation", Example 3:
    # A (table [1, 2, 3, 6]) positions 9..12 -> 13, 14, 15, 24; B ([4, 5]) position 7 -> 23.
    g = golden("block_tables_vllm_example3.json")
    bs = g["block_size"]
    tables = np.array([[1, 2, 3, 6], [4, 5, -1, -1]], np.int32)
    got = oracle.slot_mapping_varlen(tables, np.array([0, 4, 5], np.int32), np.array([13, 8], np.int32), bs,
                                     lib=lib)
    assert got.tolist() == [13, 14, 15, 24, 23], got


ALL_CHECKS = [check_f16_decoder, check_bf16_decoder, check_f32_decoder, check_worked_slots,
              check_append_roundtrip, check_bruteforce, check_closed_forms,
              check_relabel_and_heads, check_e4m3_decoder, check_e4m3_encoder, check_fp8_append,
              check_fp8_attention, check_prefill_vs_torch_sdpa, check_prefill_bruteforce_with_context,
              check_prefill_chunking_and_decode, check_fp8_prefill, check_varlen_slots]
