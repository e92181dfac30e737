"""The seeded input generator (CPU only)."""
import numpy as np

from dense_gemm_tensor_tcgen05_gb300 import inputs


def test_splitmix64_published_sequence():
    # SplitMix64 seeded with 0: the first outputs of the published generator.
    got = inputs.splitmix64(0, 0, 3)
    assert [int(x) for x in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_slices_agree():
    whole = inputs.splitmix64(12345, 0, 1000)
    part = inputs.splitmix64(12345, 600, 50)
    assert np.array_equal(whole[600:650], part)


def test_uniform_range_and_grid():
    x = inputs.uniform_f32(1, 0, (300, 400))
    assert x.dtype == np.float32 and x.min() >= -1.0 and x.max() < 1.0
    # every value is k / 2^23 - 1 for an integer k
    k = (x.astype(np.float64) + 1.0) * 2 ** 23
    assert np.array_equal(k, np.round(k))
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1 / np.sqrt(3)) < 0.01


def test_normal_moments():
    x = inputs.normal_f32(2, 1, (1000, 1000), sigma=0.25)
    assert abs(float(x.mean())) < 2e-3
    assert abs(float(x.std()) - 0.25) < 2e-3


def test_seed_and_matrix_id_separate_streams():
    a = inputs.make("uniform", "f16", 8, 8, 7, 0)
    b = inputs.make("uniform", "f16", 8, 8, 7, 1)
    a2 = inputs.make("uniform", "f16", 8, 8, 7, 0)
    assert np.array_equal(a, a2) and not np.array_equal(a, b)


def test_bf16_round_to_nearest_even():
    w = np.array([0x3F808000,   # exactly half way, even neighbour 0x3F80
                  0x3F818000,   # exactly half way, even neighbour 0x3F82
                  0x3F808001,   # just above half way
                  0x3F807FFF,   # just below half way
                  0xBF818000],  # negative tie -> even
                 dtype=np.uint32)
    got = inputs.round_to_bf16_bits(w.view(np.float32))
    assert [int(v) for v in got] == [0x3F80, 0x3F82, 0x3F81, 0x3F80, 0xBF82]


def test_f16_round_to_nearest_even():
    # 1 + 2^-11 is half way between 1 and 1 + 2^-10 -> even (1.0)
    x = np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11], dtype=np.float32)
    assert [int(v) for v in inputs.round_to_f16_bits(x)] == [0x3C00, 0x3C02]


def test_small_int_pattern_values():
    a = inputs.make("small_int", "f32", 3, 4, 0, 0)
    b = inputs.make("small_int", "f32", 3, 4, 0, 1)
    assert a.tolist() == [[-3, -1, 1, 3], [-2, 0, 2, -3], [-1, 1, 3, -2]]
    assert b.tolist() == [[-2, -1, 0, 1], [1, 2, -2, -1], [-1, 0, 1, 2]]


def test_padding_is_poisoned():
    x = inputs.make("uniform", "bf16", 3, 5, 0, 0)
    p = inputs.padded(x, 8)
    assert np.array_equal(p[:, :5], x) and np.all(p[:, 5:] == 0x7BFF)
