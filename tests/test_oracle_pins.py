"""The oracle against its pins, and planted mistakes against the pins.

Every pin is described in oracle_pins.py.  The second test copies the oracle's
C source, plants one plausible mistake (a wrong index, a dropped term, a sign,
a transposed operand), builds the copy and checks that at least one pin fails.
"""
import pytest

import oracle
from oracle_pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle.load())


MUTATIONS = [
    ("slot_off_by_one", "return blk * block_size + pos % block_size;",
     "return blk * block_size + pos % block_size + 1;"),
    ("head_map_modulo", "int h = g / G;", "int h = g % J->hkv;"),
    ("in_block_offset", "int64_t off = t % J->bs;", "int64_t off = (t + 1) % J->bs;"),
    ("table_index", "+ t / J->bs];\n            if (blk < 0 || blk >= J->num_blocks) { J->status = -1; blk = 0; }\n            int64_t off",
     "+ t % J->bs];\n            if (blk < 0 || blk >= J->num_blocks) { J->status = -1; blk = 0; }\n            int64_t off"),
    ("prefill_table_index", "+ t / J->bs];\n            if (blk < 0 || blk >= J->num_blocks) { J->status = -1; blk = 0; }\n            size_t base",
     "+ t % J->bs];\n            if (blk < 0 || blk >= J->num_blocks) { J->status = -1; blk = 0; }\n            size_t base"),
    ("score_sign", "x[t] = J->scale * acc;", "x[t] = -J->scale * acc;"),
    ("no_max_subtraction", "x[t] = exp(x[t] - mx);", "x[t] = exp(x[t]);"),
    ("no_normalisation", "double w = x[t] / sum;", "double w = x[t];"),
    ("last_token_dropped", "for (int t = 0; t < n; ++t) {\n            double w",
     "for (int t = 0; t + 1 < n; ++t) {\n            double w"),
    ("keys_as_values", "o[d] += w * V[", "o[d] += w * K["),
    ("q_row_of_kv_head", "qd[d] = orc_load(J->q, (size_t)r * D + d, J->q_dtype);\n        /* 2. scores */",
     "qd[d] = orc_load(J->q, ((size_t)s * J->hq + h) * D + d, J->q_dtype);\n        /* 2. scores */"),
    ("append_transposed_layout",
     "size_t dst = (size_t)(((blk * num_kv_heads + h) * block_size + off)) * row;",
     "size_t dst = (size_t)(((blk * block_size + off) * num_kv_heads + h)) * row;"),
    ("half_subnormal_exponent", "v = ldexp((double)frac, -24);", "v = ldexp((double)frac, -25);"),
    ("bf16_shift", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("e4m3_bias", "v = ldexp((double)(8 + frac), expo - 10);", "v = ldexp((double)(8 + frac), expo - 11);"),
    ("e4m3_subnormal", "v = ldexp((double)frac, -9);", "v = ldexp((double)frac, -10);"),
    ("e4m3_ties_odd", "(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    ("e4m3_ties_away", "(err == best_err && (c & 1) == 0)", "(err == best_err)"),
    ("e4m3_overflow_nan", "if (a >= 448.0) return sign | 0x7e;", "if (a >= 464.0) return sign | 0x7f;"),
    ("e4m3_sign_dropped", "return sign | (uint8_t)best;", "return (uint8_t)best;"),
    ("quantize_multiplies", "float y = x / scale;", "float y = x * scale;"),
    ("append_v_with_k_scale", "head_dim, v_scale, v_cache + dst);", "head_dim, k_scale, v_cache + dst);"),
    ("attention_k_with_v_scale", "K[(size_t)t * D + d] = J->k_scale *", "K[(size_t)t * D + d] = J->v_scale *"),
    ("attention_v_unscaled", "V[(size_t)t * D + d] = J->v_scale *", "V[(size_t)t * D + d] = 1.0 *"),
    ("prefill_excludes_own_token", "int last = J->ctx[s] - n + i; /* position", "int last = J->ctx[s] - n + i - 1; /* position"),
    ("prefill_no_context_offset", "int last = J->ctx[s] - n + i; /* position", "int last = i; /* position"),
    ("prefill_no_causal_mask", "int last = J->ctx[s] - n + i; /* position", "int last = J->ctx[s] - 1; /* position"),
    ("prefill_head_modulo", "int g = (int)(r % J->hq), h = g / G;", "int g = (int)(r % J->hq), h = g % J->hkv;"),
    ("varlen_slot_offset", "context_lens[s] - n + i, block_size);", "context_lens[s] - n + i + 1, block_size);"),
    ("prefill_k_with_v_scale", "acc += qd[d] * (J->k_scale * orc_load(J->k_cache",
     "acc += qd[d] * (J->v_scale * orc_load(J->k_cache"),
    ("prefill_v_unscaled", "o[d] += w * (J->v_scale * orc_load(J->v_cache", "o[d] += w * (1.0 * orc_load(J->v_cache"),
    ("prefill_q_read_as_cache_type", "qd[d] = orc_load(J->q, (size_t)r * D + d, J->q_dtype);\n        double mx",
     "qd[d] = orc_load(J->q, (size_t)r * D + d, J->kv_dtype);\n        double mx"),
]


# Anchors that occur in both the decode and the multi-token code: (name, old,
# new, occurrence), the occurrence counted from the top of the source (the
# decode function comes first).
SHARED = [
    ("score_sign", "x[t] = J->scale * acc;", "x[t] = -J->scale * acc;"),
    ("no_max_subtraction", "x[t] = exp(x[t] - mx);", "x[t] = exp(x[t]);"),
    ("no_normalisation", "double w = x[t] / sum;", "double w = x[t];"),
]
MUTATIONS = [m for m in MUTATIONS if m[0] not in {x[0] for x in SHARED}]
MUTATIONS = [m + (0,) for m in MUTATIONS] + [m + (0,) for m in SHARED] + \
    [("prefill_" + m[0], m[1], m[2], 1) for m in SHARED]


def _replace_nth(src, old, new, nth):
    pos = -1
    for _ in range(nth + 1):
        pos = src.index(old, pos + 1)
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, nth, tmp_path):
    with open(oracle.SOURCE) as f:
        src = f.read()
    expect = 2 if any(name.endswith(m[0]) for m in SHARED) else 1
    assert src.count(old) == expect, f"mutation anchor for {name} occurs {src.count(old)} times"
    path = tmp_path / "mutant.c"
    path.write_text(_replace_nth(src, old, new, nth))
    lib = oracle.load(oracle.build(str(path), str(tmp_path / "libmutant.so"), force=True))
    caught = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError) as exc:  # a mutant may also fail its own checks
            caught.append((check.__name__, type(exc).__name__))
    assert caught, f"planted mistake {name} passed every pin"
