"""Pins of the NVFP4 weight format (oracle.decode_nvfp4 / synthetic.quantize_nvfp4),
the 4-bit weights of the OCRia-1 inference stack ("OCRia-1 technical report
guide", inference stack), against the format's own definition: the 16 E2M1
values, round-to-nearest-even with saturation, one E4M3 scale per 16
consecutive elements of a row times one float32 tensor scale, and the
quantisation error that grid allows."""
import numpy as np

import oracle
import synthetic as syn

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_code_table():
    vals = oracle.decode_e2m1(np.arange(16))
    assert list(vals[:8]) == E2M1
    assert list(vals[8:]) == [-v for v in E2M1]
    assert np.signbit(vals[8])                          # code 8 is -0


def test_e2m1_rounding_ties_to_even_and_saturates():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.25, -5.0, 0.26, 4.9, 5.1], np.float32)
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, 0.0, -4.0, 0.5, 4.0, 6.0]
    got = oracle.decode_e2m1(syn.f32_to_e2m1(x))
    assert list(got) == want
    c = np.arange(16, dtype=np.uint8)
    back = syn.f32_to_e2m1(oracle.decode_e2m1(c))
    assert list(back) == [int(v) if v != 8 else 0 for v in c]   # every value round-trips (-0 -> +0)


def test_block_scale_groups_sixteen_elements_of_a_row():
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 16, (3, 64)).astype(np.uint8)
    bs = rng.integers(0x30, 0x50, (3, 4)).astype(np.uint8)        # positive normal e4m3 scales
    v = oracle.decode_nvfp4(codes, bs, 0.125)
    ref = oracle.decode_e2m1(codes).astype(np.float64) * np.repeat(oracle.decode_e4m3(bs), 16, axis=1) * 0.125
    np.testing.assert_array_equal(v, ref.astype(np.float32))
    bs2 = bs.copy()
    bs2[1, 2] += 1                                                  # one block of one row
    diff = oracle.decode_nvfp4(codes, bs2, 0.125) != v
    assert not diff[[0, 2]].any() and not diff[1, :32].any() and not diff[1, 48:].any()


def test_quantisation_error_within_the_grid():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((16, 256)) * rng.uniform(0.01, 3.0, (16, 1))).astype(np.float32)
    codes, bs, ts = syn.quantize_nvfp4(w)
    assert codes.shape == w.shape and bs.shape == (16, 16) and codes.max() < 16
    q = oracle.decode_nvfp4(codes, bs, ts)
    blk = np.abs(w).reshape(16, 16, 16).max(-1)
    err = np.abs(q - w).reshape(16, 16, 16).max(-1)
    # E2M1's widest step (4 -> 6) is 1/3 of the block maximum 6: half of it plus the scale's
    # E4M3 rounding (3 mantissa bits) bounds the error by about a fifth of the block maximum
    assert (err <= 0.21 * blk + 1e-12).all()
    assert np.abs(q - w).mean() < 0.12 * np.abs(w).mean()      # about 9% for Gaussian rows
    # the tensor scale puts the largest block scale at the top of the E4M3 range
    assert abs(ts - np.abs(w).max() / (6 * 448)) <= 1e-6 * ts
