"""Pins for the oracle's output codecs (bf16, FP8 e4m3).

Each encoder is checked against (a) the format definition exhaustively over
all codes and (b) torch's own float8_e4m3fn / bfloat16 conversions, a library
routine independent of the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import codecs


def _torch_e4m3_codes(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_table_endpoints():
    vals = codecs.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert vals[0x00] == 0.0
    assert vals[0x01] == 2.0 ** -9                     # smallest subnormal
    assert vals[0x07] == 7 * 2.0 ** -9                 # largest subnormal
    assert vals[0x08] == 2.0 ** -6                     # smallest normal
    assert vals[0x38] == 1.0                           # exponent field 7 = bias
    assert vals[0x7E] == 448.0                         # largest finite
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert vals[0xFE] == -448.0
    assert np.signbit(vals[0x80]) and vals[0x80] == 0.0


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = codecs.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))


def test_e4m3_roundtrip_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = codecs.e4m3_encode(codecs.e4m3_decode(codes))
    # -0 and +0 keep their sign
    assert np.array_equal(back, codes)


def test_e4m3_ties_to_even_at_every_midpoint():
    pos = np.array([c for c in range(0x7E + 1)], dtype=np.uint8)
    v = codecs.e4m3_decode(pos)
    mids = (v[:-1] + v[1:]) / 2.0
    got = codecs.e4m3_encode(mids)
    lo, hi = pos[:-1], pos[1:]
    expect = np.where((lo & 1) == 0, lo, hi)
    assert np.array_equal(got, expect)
    got_neg = codecs.e4m3_encode(-mids)
    assert np.array_equal(got_neg, expect | 0x80)


def test_e4m3_saturates():
    for y in [448.0, 449.0, 464.0, 480.0, 1e6, np.inf]:
        assert codecs.e4m3_encode(np.array([y]))[0] == 0x7E
        assert codecs.e4m3_encode(np.array([-y]))[0] == 0xFE


def test_e4m3_matches_torch_within_range():
    rng = np.random.default_rng(1)
    # every float32 value on a dense grid in [-448, 448] plus random magnitudes over all binades
    grid = np.linspace(-448.0, 448.0, 200001).astype(np.float32)
    rnd = (rng.choice([-1, 1], 200000) * np.exp2(rng.uniform(-12, 8.8, 200000))).astype(np.float32)
    x = np.concatenate([grid, rnd])
    x = x[np.abs(x) <= 448.0]
    assert np.array_equal(codecs.e4m3_encode(x.astype(np.float64)), _torch_e4m3_codes(x))


def test_bf16_matches_torch_on_float32_patterns():
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 2 ** 32, 400000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = codecs.bf16_bits(x.astype(np.float64))
    assert np.array_equal(ours, ref)


def test_bf16_ties_to_even():
    # 1 + 2**-8 sits halfway between 1 and 1 + 2**-7: even mantissa (1.0) wins;
    # 1 + 3 * 2**-8 sits between 1 + 2**-7 and 1 + 2**-6: even (1 + 2**-6) wins.
    assert codecs.bf16_round(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert codecs.bf16_round(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    # just above the midpoint rounds up (a float64-only value: no float32 pre-rounding)
    assert codecs.bf16_round(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1 + 2.0 ** -7


def test_bf16_overflow_and_subnormals():
    assert codecs.bf16_round(np.array([codecs.BF16_MAX]))[0] == codecs.BF16_MAX
    assert np.isinf(codecs.bf16_round(np.array([2.0 ** 128]))[0])
    assert codecs.bf16_round(np.array([2.0 ** -133]))[0] == 2.0 ** -133
    assert codecs.bf16_round(np.array([2.0 ** -135]))[0] == 0.0


@pytest.mark.parametrize("planted", ["floor", "short_mantissa"])
def test_planted_codec_mistakes_are_caught(monkeypatch, planted):
    """A plausible mistake in the encoder fails the library comparison."""
    if planted == "floor":
        monkeypatch.setattr(codecs.np, "rint", np.floor)
    else:
        orig = codecs._round_to_grid
        monkeypatch.setattr(codecs, "_round_to_grid",
                            lambda x, m, e: orig(x, m - 1, e))
    x = np.linspace(-448.0, 448.0, 20001).astype(np.float32)
    x = np.concatenate([x, np.float32([3e-3, -5e-3, 1.5e-3])])
    ours = codecs.e4m3_encode(x.astype(np.float64))
    assert not np.array_equal(ours, _torch_e4m3_codes(x))
