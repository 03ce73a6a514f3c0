"""GPU: w4a16_pack / w4a16_unpack are bit-exact against the oracle's packer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from oracle import w4a16_oracle as O  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("R,C", [(8, 1), (8, 8), (64, 24), (40, 4), (16, 3), (1024, 776), (5376, 520)])
def test_pack_rows_bit_exact(R, C):
    rng = np.random.default_rng(R * 7 + C)
    codes = rng.integers(0, 16, size=(R, C), dtype=np.uint8)
    got = w4.pack(torch.from_numpy(codes).cuda(), dim=0).cpu().numpy()
    assert np.array_equal(got, O.pack_rows(codes))
    back = w4.unpack(torch.from_numpy(got).cuda(), dim=0).cpu().numpy()
    assert np.array_equal(back, codes)


@pytest.mark.parametrize("R,C", [(1, 8), (3, 16), (168, 43008 // 8), (2, 776), (16, 8)])
def test_pack_cols_bit_exact(R, C):
    rng = np.random.default_rng(R * 13 + C)
    codes = rng.integers(0, 16, size=(R, C), dtype=np.uint8)
    got = w4.pack(torch.from_numpy(codes).cuda(), dim=1).cpu().numpy()
    assert np.array_equal(got, O.pack_cols(codes))
    back = w4.unpack(torch.from_numpy(got).cuda(), dim=1).cpu().numpy()
    assert np.array_equal(back, codes)


def test_golden_words_on_device(golden):
    for row in golden("pack_words.txt"):
        kind, codes, word = row[0], np.array([int(v) for v in row[1:9]], dtype=np.uint8), int(row[9], 16)
        t = torch.from_numpy(codes.reshape((1, 8) if kind == "cols" else (8, 1))).cuda()
        got = w4.pack(t, dim=1 if kind == "cols" else 0).cpu().numpy().view(np.uint32)
        assert int(got.ravel()[0]) == word, (kind, codes)


def test_unpack_negative_words():
    w = np.array([[-1, -2147483648, 0x12345678, -559038737]], dtype=np.int32)
    for dim in (0, 1):
        got = w4.unpack(torch.from_numpy(w).cuda(), dim=dim).cpu().numpy()
        want = O.unpack_rows(w) if dim == 0 else O.unpack_cols(w)
        assert np.array_equal(got, want)


def test_pack_uses_low_nibble_only():
    codes = np.array([[0x1F, 0x2E, 0x3D, 0x4C, 0x5B, 0x6A, 0x79, 0x88]], dtype=np.uint8)
    got = w4.pack(torch.from_numpy(codes).cuda(), dim=1).cpu().numpy()
    assert np.array_equal(got, O.pack_cols(codes & 0xF))
