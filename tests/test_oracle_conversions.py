"""Pins for the oracle's element conversions, against library routines.

The gather's dequant path is fp32(e4m3(x)) * scale rounded once to the
destination type ("MLA cache gather scheduled per logical page", section
"实现拆解" item 1: FP8 -> BF16 while copying). The page fixes neither the
FP8 variant nor the rounding; the oracle reads them as OCP E4M3 ("fn") and
round-to-nearest-even. These tests tie the oracle's own decoders and
encoders, written from the format definitions, to torch's and numpy's casts:
a wrong bias, a dropped subnormal branch or a round-half-up would fail here.
"""
import numpy as np
import pytest
import torch

from oracle import gather as og


def _same_bits_or_both_nan(a_bits: np.ndarray, b_bits: np.ndarray, nan_of) -> None:
    a_nan = nan_of(a_bits)
    b_nan = nan_of(b_bits)
    assert np.array_equal(a_nan, b_nan)
    keep = ~a_nan
    bad = np.nonzero(a_bits[keep] != b_bits[keep])[0]
    assert bad.size == 0, f"{bad.size} mismatches, first: {a_bits[keep][bad[:5]]} vs {b_bits[keep][bad[:5]]}"


def _bf16_nan(bits):
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def _f16_nan(bits):
    return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x03FF) != 0)


def _f32_nan(bits):
    return ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x007FFFFF) != 0)


def test_e4m3_decode_all_256_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = np.array([og.e4m3_to_f32(int(c)) for c in codes], dtype=np.float32)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    _same_bits_or_both_nan(ours.view(np.uint32), ref.view(np.uint32), _f32_nan)
    # the format's landmarks: max 448, smallest subnormal 2^-9, NaN only at S.1111.111
    assert og.e4m3_to_f32(0x7E) == 448.0
    assert og.e4m3_to_f32(0x01) == 2.0 ** -9
    assert og.e4m3_to_f32(0x08) == 2.0 ** -6
    assert np.isnan(og.e4m3_to_f32(0x7F)) and np.isnan(og.e4m3_to_f32(0xFF))
    assert np.signbit(og.e4m3_to_f32(0x80)) and og.e4m3_to_f32(0x80) == 0.0


def test_bf16_and_f16_decode_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ours_bf = og.convert_array(codes, "bf16", "fp32")
    ref_bf = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float32).numpy().view(np.uint32)
    _same_bits_or_both_nan(ours_bf, ref_bf, _f32_nan)
    ours_h = og.convert_array(codes, "fp16", "fp32")
    ref_h = codes.view(np.float16).astype(np.float32).view(np.uint32)
    _same_bits_or_both_nan(ours_h, ref_h, _f32_nan)


def _f32_specials():
    vals = [0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 3.4028235e38, -3.4028235e38,
            1.1754944e-38, 1e-45, -1e-45, 65504.0, 65519.99, 65520.0, 6.1035156e-05, 5.9604645e-08,
            2.9802322e-08, 2.9802326e-08, 1.0 + 2.0 ** -8, 1.0 + 2.0 ** -7 + 2.0 ** -8, 1.0 + 2.0 ** -11,
            1.0 + 3 * 2.0 ** -11]
    bits = np.array(vals, dtype=np.float32).view(np.uint32)
    # exact ties for bf16 (low 16 bits = 0x8000) with even and odd kept bit
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x7F7F8000, 0x00018000, 0x00008000], dtype=np.uint32)
    return np.concatenate([bits, ties])


@pytest.mark.parametrize("seed", [0, 1])
def test_f32_to_bf16_rne_matches_torch(seed):
    rng = np.random.default_rng(seed)
    bits = np.concatenate([rng.integers(0, 2 ** 32, 300_000, dtype=np.uint64).astype(np.uint32), _f32_specials()])
    ours = np.fromiter((og.f32_to_bf16(float(x)) for x in bits.view(np.float32)), dtype=np.uint16,
                       count=bits.shape[0])
    ref = torch.from_numpy(bits.view(np.float32).copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    _same_bits_or_both_nan(ours, ref, _bf16_nan)


@pytest.mark.parametrize("seed", [0, 1])
def test_f32_to_f16_rne_matches_numpy(seed):
    rng = np.random.default_rng(100 + seed)
    # bias the exponent toward binary16's range (and its subnormals) so that
    # rounding at every shift is exercised, plus fully random patterns
    sign = rng.integers(0, 2, 300_000, dtype=np.uint32) << 31
    exp = rng.integers(127 - 30, 127 + 17, 300_000, dtype=np.uint32) << 23
    man = rng.integers(0, 2 ** 23, 300_000, dtype=np.uint32)
    near = sign | exp | man
    bits = np.concatenate([near, rng.integers(0, 2 ** 32, 100_000, dtype=np.uint64).astype(np.uint32),
                           _f32_specials()])
    ours = np.fromiter((og.f32_to_f16(float(x)) for x in bits.view(np.float32)), dtype=np.uint16,
                       count=bits.shape[0])
    with np.errstate(over="ignore"):
        ref = bits.view(np.float32).astype(np.float16).view(np.uint16)
    _same_bits_or_both_nan(ours, ref, _f16_nan)


@pytest.mark.parametrize("scale", [1.0, 0.05, 0.02, 2.0 ** -12, 1e30, 3.0e-39])
@pytest.mark.parametrize("dst", ["bf16", "fp16", "fp32"])
def test_e4m3_dequant_all_codes_all_targets(scale, dst):
    """fp32(e4m3) * scale (one fp32 multiply) rounded to the target, against torch."""
    codes = np.arange(256, dtype=np.uint8)
    ours = og.convert_array(codes, "fp8_e4m3", dst, scale)
    prod = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32) * torch.tensor(scale, dtype=torch.float32)
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dst]
    ref = prod.to(tdt)
    ref_bits = ref.view({"bf16": torch.int16, "fp16": torch.int16, "fp32": torch.int32}[dst]).numpy()
    ref_bits = ref_bits.view({"bf16": np.uint16, "fp16": np.uint16, "fp32": np.uint32}[dst])
    nan_of = {"bf16": _bf16_nan, "fp16": _f16_nan, "fp32": _f32_nan}[dst]
    _same_bits_or_both_nan(ours, ref_bits, nan_of)


def test_supported_pairs():
    ok = {("bf16", "bf16"), ("fp16", "fp16"), ("fp32", "fp32"), ("fp8_e4m3", "fp8_e4m3"), ("u8", "u8"),
          ("fp8_e4m3", "bf16"), ("fp8_e4m3", "fp16"), ("fp8_e4m3", "fp32"), ("bf16", "fp32"), ("fp16", "fp32")}
    names = list(og.DTYPE_CODES)
    for s in names:
        for d in names:
            assert og.pair_supported(s, d) == ((s, d) in ok), (s, d)
