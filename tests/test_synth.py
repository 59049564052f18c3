"""The seeded input generator (no GPU)."""
import numpy as np

import synth


def test_splitmix64_reference_outputs():
    # The published SplitMix64 reference sequence for seed 1234567.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(v) for v in synth.splitmix64(1234567, 0, 5)] == want


def test_values_depend_only_on_seed_stream_index():
    a = synth.normal_f32(1, 3, 1e-3, 0, 300_001)
    b = synth.normal_f32(1, 3, 1e-3, 123, 1000)
    np.testing.assert_array_equal(a[123:1123], b)
    idx = np.array([0, 1, 2, 99_999, 300_000])
    np.testing.assert_array_equal(a[idx], synth.normal_f32_at(1, 3, 1e-3, idx))
    # thread count does not change the values
    c = np.empty(300_001, np.float32)
    synth.fill_normal_f32(c.ctypes.data, 1, 3, 1e-3, 0, 300_001, threads=1)
    np.testing.assert_array_equal(a, c)
    t = synth.student_t3_bf16(3, 2, 1e-3, 0, 200_000)
    np.testing.assert_array_equal(t[idx[:4]], synth.student_t3_bf16_at(3, 2, 1e-3, idx[:4]))
    # different streams differ
    assert not np.array_equal(a[:100], synth.normal_f32(1, 4, 1e-3, 0, 100))


def test_distributions():
    z = synth.normal_f32(7, 0, 2.0, 0, 2_000_000).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 2.0) < 0.01
    t = synth.student_t3_f32(7, 1, 1.0, 0, 2_000_000).astype(np.float64)
    # Student-t with 3 degrees of freedom: median 0, quartiles +-0.7649,
    # P(|T| > 3.182) = 0.05
    q1, q3 = np.quantile(t, [0.25, 0.75])
    assert abs(q1 + 0.7649) < 0.01 and abs(q3 - 0.7649) < 0.01
    assert abs(np.mean(np.abs(t) > 3.182) - 0.05) < 0.002
    tb = synth.student_t3_bf16(7, 1, 1.0, 0, 1000)
    assert tb.dtype == np.uint16


def test_workload_sizes():
    w = synth.WORKLOADS
    assert w["speech300m_n8_f32"].min_bytes == 2 * 8 * 300_000_000 * 4
    assert w["ring4_uneven_1m_f32"].p == 1_048_579
    assert w["transformer24_buckets_n4_f32"].p == 1_339_670_528
    assert w["resnet18_sgd_n32_f32"].p == 11_689_512
    assert w["student_t3_1g_n16_bf16"].elem_bytes == 2
