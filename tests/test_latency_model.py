"""The two-segment latency model used to fit this kernel's timings: its marginal cost
of recomputing one more block must be the paper's Eq. 5 (Fig. 6 caption),
dT_B = T(l1, q1+1, l2-1, q2) - T(l1, q1, l2, q2) = k5 (l1 + 2 q1) + (k2 - k3 + k5),
and the least-squares fit must recover known coefficients."""
import numpy as np

import bench


def T(k, l1, q1, l2, q2):
    return float(np.dot(k, bench.latency_model_terms(l1, q1, l2, q2)))


def test_model_difference_is_eq5():
    rng = np.random.default_rng(0)
    for _ in range(200):
        k = rng.standard_normal(6)
        l1, q1, l2, q2 = (int(x) for x in rng.integers(0, 500, 4))
        l2 += 1
        d = T(k, l1, q1 + 1, l2 - 1, q2) - T(k, l1, q1, l2, q2)
        assert abs(d - (k[5] * (l1 + 2 * q1) + (k[2] - k[3] + k[5]))) < 1e-6 * (1 + abs(d))


def test_fit_recovers_known_coefficients():
    rng = np.random.default_rng(1)
    k = np.array([0.02, 1e-4, 8e-4, 2e-4, 9e-4, 3e-6])
    samples = []
    for l1 in (0, 64, 256):
        for q1 in (16, 64, 128):
            for l2 in (0, 64, 256):
                for q2 in (8, 32):
                    samples.append((l1, q1, l2, q2, T(k, l1, q1, l2, q2) * (1 + 1e-4 * rng.standard_normal())))
    kf, r2 = bench.fit_latency_model(samples)
    assert r2 > 0.9999
    np.testing.assert_allclose(kf[5], k[5], rtol=1e-2)
    np.testing.assert_allclose(kf[2], k[2], rtol=5e-2)
