"""The exact E4M3 -> f16 identity the E4M3 decode kernels use for V (and K in
the f16 Q.K^T form): an E4M3 code s.eeee.mmm read as the f16 bit pattern
s.0eeee.mmm0000000 is the code's value times 2^-8.  The kernels reach that
pattern for two codes of a 32-bit word at once, from the word's odd bytes
(bytes 1 and 3) with one shift and one logic operation, and from its even
bytes (0 and 2) after a shift by one byte.  Both forms are checked here for
every finite code, in both halves of a word and next to every other byte
value, against torch's float8_e4m3fn decode (an implementation independent
of this one)."""
import numpy as np
import torch


def odd_bytes(r: np.ndarray) -> np.ndarray:
    r = r.astype(np.uint32)
    return ((r >> 1) & 0x3F803F80) | (r & 0x80008000)


def even_bytes(r: np.ndarray) -> np.ndarray:
    return odd_bytes((r.astype(np.uint64) << 8).astype(np.uint32))


def _halves(out):
    lo = (out & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    hi = (out >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    return lo, hi


def _decode(codes) -> np.ndarray:
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_every_finite_code_in_both_halves_next_to_any_byte():
    codes = np.arange(256, dtype=np.uint32)
    finite = (codes & 0x7F) != 0x7F  # 0x7F / 0xFF are NaN in E4M3
    ref = _decode(codes) * 2.0 ** -8
    for other in (0x00, 0x3C, 0xC1, 0x7E, 0x80, 0xFF):  # the code converted in the other half
        o = np.uint32(other)
        o_ref = _decode([other])[0] * 2.0 ** -8 if (other & 0x7F) != 0x7F else None
        for junk in (0x00, 0xFF, 0x5A):  # the bytes each form ignores
            j = np.uint32(junk)
            # odd bytes: the code in byte 1 (low half) and `other` in byte 3
            lo, hi = _halves(odd_bytes((codes << 8) | (o << 24) | j | (j << 16)))
            np.testing.assert_array_equal(lo[finite], ref[finite])
            if o_ref is not None:
                assert np.all(hi == o_ref)
            # even bytes: the code in byte 0 and `other` in byte 2
            lo, hi = _halves(even_bytes(codes | (o << 16) | (j << 8) | (j << 24)))
            np.testing.assert_array_equal(lo[finite], ref[finite])
            if o_ref is not None:
                assert np.all(hi == o_ref)


def test_signed_zero_and_no_crossing_between_halves():
    # The sign of zero survives, and a code's bits never reach the other half.
    assert odd_bytes(np.array([0x80008000], dtype=np.uint32))[0] == 0x80008000
    assert even_bytes(np.array([0x00800080], dtype=np.uint32))[0] == 0x80008000
    assert odd_bytes(np.array([0x7F00FF00], dtype=np.uint32))[0] >> 16 == 0x3F80
    assert even_bytes(np.array([0x00FF007F], dtype=np.uint32))[0] & 0xFFFF == 0x3F80
