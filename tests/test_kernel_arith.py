"""The bit-level dequantisation steps of the tensor-core kernels, emulated on
the host and checked against the weight formats' definitions (CPU).

The prefill kernels turn quantised weights into bf16 tensor-core operands with
integer and bf16 operations whose correctness rests on facts about the
formats; these tests check those facts for every code:
- MX (OCP E4M3 / E2M1 with an E8M0 scale 2^(s-127)): the hardware widens a
  code to fp16 exactly; moving the fp16 exponent field into the low bits of
  the bf16 one gives the element times 2^-112; one bf16 multiply by the bf16
  whose bits are (s + 112) << 7, i.e. 2^(s-15), then gives the weight
  element * 2^(s-127), exactly whenever that value is a bf16 (the fast range
  s <= 142).
- int4 g128: the nibble pair trick ((nibble ^ 8) in the low mantissa bits of
  the bf16 128) gives 136 + q; subtracting 136 is exact; the multiply by the
  group scale rounds q * s once to bf16.
"""
import numpy as np
import pytest
import torch


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (the tensor-core operand)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def e4m3_values() -> tuple:
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    keep = ~np.isnan(vals)
    return codes[keep], vals[keep]


def e2m1_values() -> tuple:
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # E2M1: bias 1, one mantissa bit
    codes = np.arange(16, dtype=np.uint8)
    vals = np.array([(-1.0 if c & 8 else 1.0) * mags[c & 7] for c in codes])
    return codes, vals


def shifted_bf16(values: np.ndarray) -> np.ndarray:
    """fp16 bits of the (exactly widened) elements -> the kernel's bf16 bits:
    ((h & 0x7FFF) >> 3) | (h & 0x8000)."""
    h = values.astype(np.float16)
    assert np.array_equal(h.astype(np.float64), values)  # the widening is exact
    hb = h.view(np.uint16).astype(np.uint32)
    return (((hb & 0x7FFF) >> 3) | (hb & 0x8000)).astype(np.uint16)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_mx_shifted_elements_are_exact(fmt):
    codes, vals = e4m3_values() if fmt == "e4m3" else e2m1_values()
    got = bf16_bits_to_f32(shifted_bf16(vals)).astype(np.float64)
    assert np.array_equal(got, vals * 2.0 ** -112)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_mx_fast_conversion_gives_the_weight(fmt):
    """For every code and every scale of the fast range, one bf16 multiply of
    the shifted element by the bf16 with bits (s + 112) << 7 equals the weight
    element * 2^(s-127) rounded to bf16, and equals it exactly whenever the
    weight is a bf16 normal or zero."""
    codes, vals = e4m3_values() if fmt == "e4m3" else e2m1_values()
    x = bf16_bits_to_f32(shifted_bf16(vals))
    for s in range(0, 143):
        fac = bf16_bits_to_f32(np.array([(s + 112) << 7], dtype=np.uint16))[0]
        assert float(fac) == 2.0 ** (s - 15)
        # the bf16 FMA computes x * fac + (-0) exactly, then rounds once
        prod = (x.astype(np.float64) * float(fac))
        got = f32_to_bf16_rne(prod.astype(np.float32))
        want_exact = vals * 2.0 ** (s - 127)
        want = f32_to_bf16_rne(want_exact.astype(np.float32))
        assert np.array_equal(got, want), s
        normal = (np.abs(want_exact) >= 2.0 ** -126) | (want_exact == 0)
        back = bf16_bits_to_f32(got).astype(np.float64)
        assert np.array_equal(back[normal], want_exact[normal]), s


def test_mx_fast_range_ends_at_scale_142():
    """2^(s-15) is a bf16 normal up to s = 142 (bf16 exponent field 254); the
    scale 143 would need field 255 (inf): such layers take the fp32 path."""
    assert (142 + 112) == 254
    assert bf16_bits_to_f32(np.array([(142 + 112) << 7], dtype=np.uint16))[0] == 2.0 ** 127
    assert np.isinf(bf16_bits_to_f32(np.array([(143 + 112) << 7], dtype=np.uint16))[0])


def test_int4_nibble_trick_and_group_scale():
    """(nibble ^ 8) | 0x4300 is the bf16 136 + q for the two's-complement
    nibble q; 136 + q - 136 = q exactly; q * s then rounds once to bf16."""
    nib = np.arange(16, dtype=np.uint32)
    q = np.where(nib >= 8, nib.astype(np.int64) - 16, nib.astype(np.int64))
    bits = ((nib & 0xF) ^ 0x4308).astype(np.uint16)  # the kernel's LOP3 per half
    v136 = bf16_bits_to_f32(bits).astype(np.float64)
    assert np.array_equal(v136, 136.0 + q)
    assert np.array_equal(v136 - 136.0, q.astype(np.float64))
    rng = np.random.default_rng(3)
    scales = f32_to_bf16_rne(rng.standard_normal(512).astype(np.float32) * 0.003)
    s = bf16_bits_to_f32(scales).astype(np.float64)
    prod = np.outer(s, q.astype(np.float64))  # exact: at most 12 significant bits
    got = bf16_bits_to_f32(f32_to_bf16_rne(prod.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, rne_8_bits(prod))


def rne_8_bits(x: np.ndarray) -> np.ndarray:
    """Round to 8 significant bits, ties to even (bf16 for normal values),
    written from the definition: x = m * 2^e with 0.5 <= |m| < 1."""
    out = np.zeros_like(x)
    nz = x != 0
    m, e = np.frexp(x[nz])
    out[nz] = np.ldexp(np.round(m * 256.0) / 256.0, e)  # np.round: half to even
    return out


def test_rne_8_bits_pins():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1) wins;
    # 1 + 3 * 2^-8 ties between 1 + 2^-7 and 1 + 2^-6: even (1 + 2^-6) wins
    assert rne_8_bits(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert rne_8_bits(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert rne_8_bits(np.array([-(1 + 3 * 2.0 ** -8)]))[0] == -(1 + 2.0 ** -6)
    assert rne_8_bits(np.array([255.0]))[0] == 255.0
    assert rne_8_bits(np.array([257.0]))[0] == 256.0  # 9 bits: tie to even
