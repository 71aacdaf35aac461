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


def test_packed_record_layout():
    """Two codes per byte, element 2j in the low nibble of byte j, row after
    row, then the block scales: a literal 2 x 32 record."""
    codes = np.array([[(j % 16) for j in range(32)], [(15 - j % 16) for j in range(32)]], np.uint8)
    bs = np.array([[0x38, 0x40], [0x30, 0x48]], np.uint8)
    rec = syn.pack_nvfp4(codes, bs)
    row0 = [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE] * 2
    row1 = [0xEF, 0xCD, 0xAB, 0x89, 0x67, 0x45, 0x23, 0x01] * 2
    assert list(rec) == row0 + row1 + [0x38, 0x40, 0x30, 0x48]
    assert len(rec) == syn.nvfp4_bytes(2, 32)
    c2, b2 = oracle.unpack_nvfp4(rec, 2, 32)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(b2, bs)


def test_model_weights_decode_near_their_draws():
    """An nvfp4 model's decoded matrices lie within the grid's error bound of
    the same N(0, 0.02) draws the bf16 model rounds, expert by expert (each
    expert has its own tensor scale), and the LM head and router stay bf16."""
    cfg16 = syn.scaled(syn.MOE3B, name="m16", n_layers=1, hidden=256, n_q_heads=2, n_kv_heads=2, head_dim=64,
                       n_experts=4, top_k=2, n_shared=1, inter=128, vocab=512)
    cfg4 = syn.scaled(cfg16, name="m4", wdtype=syn.NVFP4)
    w16, w4 = syn.generate_weights(cfg16, 0), syn.generate_weights(cfg4, 0)
    m16, m4 = oracle.OracleModel(w16), oracle.OracleModel(w4)
    np.testing.assert_array_equal(m16.lm_head, m4.lm_head)
    np.testing.assert_array_equal(m16.layers[0]["w_router"], m4.layers[0]["w_router"])
    for name in ("w_qkv", "w_o", "w_gate", "w_up", "w_down"):
        a, b = m16.layers[0][name], m4.layers[0][name]
        assert a.shape == b.shape
        blk = np.abs(a).reshape(-1, 16).max(-1)
        err = np.abs(b - a).reshape(-1, 16).max(-1)
        assert (err <= 0.22 * blk + 1e-6).all(), name      # the grid's bound plus the bf16 rounding of a
        assert not np.array_equal(a, b)
    s = w4.get("s_gate", 0)
    assert s.shape == (5,) and len(set(s.tolist())) == 5    # one tensor scale per expert
    w4b = syn.generate_weights(cfg4, 0)
    w4b.get("s_gate", 0)[2] *= 2
    g = oracle.OracleModel(w4b).layers[0]["w_gate"]
    np.testing.assert_array_equal(g[2], 2 * m4.layers[0]["w_gate"][2])
    np.testing.assert_array_equal(np.delete(g, 2, 0), np.delete(m4.layers[0]["w_gate"], 2, 0))
