"""The exact E4M3 -> f16 identity the E4M3 decode kernels use for V (and K in
the f16 Q.K^T form): a code in the low byte of a 16-bit half, moved up as
(y + (y & 0x80)) << 7, is the f16 bit pattern of the code's value times 2^-8.
Checked for every finite code, in both halves of a 32-bit word, against
torch's float8_e4m3fn decode (an implementation independent of this one)."""
import numpy as np
import torch


def shifted(y: np.ndarray) -> np.ndarray:
    y = y.astype(np.uint32)
    return ((y + (y & 0x00800080)) << 7) & 0xFFFFFFFF


def test_every_finite_code_in_both_halves():
    codes = np.arange(256, dtype=np.uint32)
    finite = (codes & 0x7F) != 0x7F  # 0x7F / 0xFF are NaN in E4M3
    ref = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).float().numpy()
    for lo_code in (0x00, 0x3C, 0xC1, 0x7E, 0x80):
        words = codes | (np.uint32(lo_code) << 16)  # code in the low half, another in the high half
        out = shifted(words)
        lo = (out & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
        hi = (out >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
        np.testing.assert_array_equal(lo[finite], ref[finite].astype(np.float64) * 2.0 ** -8)
        lo_ref = torch.tensor([lo_code], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
        assert np.all(hi == lo_ref * 2.0 ** -8)
    # the sign of zero survives, and no carry crosses the halves
    assert shifted(np.array([0x00800080], dtype=np.uint32))[0] == 0x80008000
