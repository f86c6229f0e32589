import numpy as np

from attn_inputs import (make_inputs, f32_to_bf16_bits, bf16_bits_to_f32, peaked_rows,
                         sweep_points, WORKLOADS)


def test_same_seed_same_bytes():
    a = make_inputs(2, 3, 17, 64, 5)
    b = make_inputs(2, 3, 17, 64, 5)
    for name in a:
        assert a[name].dtype == np.uint16 and a[name].shape == (2, 3, 17, 64)
        assert a[name].tobytes() == b[name].tobytes()


def test_tensors_are_independent_streams():
    a = make_inputs(1, 1, 64, 64, 5)
    only_v = make_inputs(1, 1, 64, 64, 5, tensors=("v",))
    assert only_v["v"].tobytes() == a["v"].tobytes()
    assert a["q"].tobytes() != a["k"].tobytes()


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -2.5, 0.0],
                 dtype=np.float32)
    r = bf16_bits_to_f32(f32_to_bf16_bits(x))
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    np.testing.assert_array_equal(r, np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 0.0], np.float32))


def test_normal_statistics():
    x = bf16_bits_to_f32(make_inputs(1, 1, 4096, 64, 9, tensors=("q",))["q"]).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_peaked_rows_scaled_by_eight():
    base = make_inputs(1, 2, 500, 16, 3, tensors=("q",))["q"]
    peaked = make_inputs(1, 2, 500, 16, 3, peaked_frac=0.01, tensors=("q",))["q"]
    rows = peaked_rows(1, 2, 500, 3, 0.01)
    assert rows.shape == (2, 5)
    a = bf16_bits_to_f32(base).reshape(2, 500, 16)
    b = bf16_bits_to_f32(peaked).reshape(2, 500, 16)
    for bh in range(2):
        mask = np.zeros(500, bool)
        mask[rows[bh]] = True
        np.testing.assert_array_equal(b[bh, mask], 8 * a[bh, mask])
        np.testing.assert_array_equal(b[bh, ~mask], a[bh, ~mask])


def test_sweep_keeps_16k_tokens():
    pts = sweep_points()
    assert len(pts) == 24
    for _, p in pts:
        assert p["B"] * p["N"] == 16384
        assert p["H"] * p["d"] == 2048
    assert WORKLOADS["long_causal_peaked"]["N"] == 32768
