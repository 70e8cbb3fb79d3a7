"""The operand splits that let 16-bit and tf32 tensor-core products reach fp32-level accuracy
(CPU, numpy emulation of the formats):
  - bf16, for the prefill's A/M products: hi = x with its low 16 bits cleared (exact in bf16),
    lo = x - hi rounded to bf16; hi*hi' + hi*lo' + lo*hi' is about 2^-16 off typically and at most
    about 2^-14 (the dropped lo*lo' term: each lo is below 2^-7 of its x);
  - tf32, for the solve and the backward: hi = x with its low 13 mantissa bits cleared, lo = x - hi
    (exact in fp32) of which the tensor core reads the top 19 bits (sign, exponent, 10 mantissa
    bits); hi*hi' + hi*lo' + lo*hi' carries about 20.
Each product of two such parts is exact in fp32, so the emulation multiplies in fp64 and only
the operand formats are modelled."""
import numpy as np


def _clear_low(x, bits):
    u = np.asarray(x, dtype=np.float32).view(np.uint32) & np.uint32((0xFFFFFFFF << bits) & 0xFFFFFFFF)
    return u.view(np.float32)


def _bf16_round(x):
    """Round-to-nearest-even to bf16 (8 significand bits), kept in fp32."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _split_bf16(x):
    hi = _clear_low(x, 16)
    return hi, _bf16_round(np.float32(x) - hi)


def _split_tf32(x):
    hi = _clear_low(x, 13)
    lo = np.float32(x) - hi  # exact in fp32
    return hi, _clear_low(lo, 13)  # what the tensor core reads of lo


def _three_term(split, x, y):
    xh, xl = split(x)
    yh, yl = split(y)
    f = lambda a: np.asarray(a, dtype=np.float64)
    return f(xh) * f(yh) + f(xh) * f(yl) + f(xl) * f(yh)


def _rel_err(split):
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    y = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    exact = x.astype(np.float64) * y.astype(np.float64)
    return np.abs(_three_term(split, x, y) - exact) / np.abs(exact)


def test_bf16_three_term_split_carries_about_16_bits():
    err = _rel_err(_split_bf16)
    assert err.max() < 2.0 ** -13 and np.median(err) < 2.0 ** -16
    # one bf16 operand alone would be off by up to 2^-8
    x = np.float32(1.0 + 2.0 ** -9 + 2.0 ** -12)
    assert abs(float(_bf16_round(x)) - float(x)) / float(x) > 2.0 ** -12


def test_tf32_three_term_split_carries_about_20_bits():
    err = _rel_err(_split_tf32)
    assert err.max() < 2.0 ** -19 and np.median(err) < 2.0 ** -21


def test_splits_keep_fp32_range():
    """Both splits keep the fp32 exponent: factors near e^{+-80} (the prefill's reference-scaled
    operands) are represented, which fp16 operands could not."""
    for split in (_split_bf16, _split_tf32):
        for x in (np.float32(np.exp(80.0)), np.float32(np.exp(-80.0))):
            hi, lo = split(x)
            assert np.isfinite(hi) and hi != 0 and abs(float(hi) + float(lo) - float(x)) <= 2.0 ** -15 * float(x)
    assert np.finfo(np.float16).max < np.exp(80.0) and np.finfo(np.float16).tiny > np.exp(-80.0)


def test_widened_bf16_values_are_exact_in_tf32():
    """A bf16 input widened to fp32 has its low 16 bits zero, so the tf32 split gives hi = x and
    lo = 0 exactly.  The backward (and nothing else) relies on it to skip the product term that would
    multiply such an operand's lo: the term adds exactly zero, and the gradients are bit-identical."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(50000) * np.exp(rng.uniform(-30, 30, 50000))).astype(np.float32)
    xb = _bf16_round(x)
    hi, lo = _split_tf32(xb)
    assert np.array_equal(hi.view(np.uint32), xb.view(np.uint32)) and np.all(lo == 0)
    # a general fp32 value is not: the split's lo carries its low mantissa bits
    h2, l2 = _split_tf32(x)
    assert np.count_nonzero(l2) > 0.99 * x.size
