"""The seeded input generators: deterministic, shaped and distributed as the workloads
state (rates of dones/truncations, truncation drawn only where not terminated)."""
import numpy as np

import synthetic_rollouts as sr


def test_deterministic_and_independent_substreams():
    a = sr.gae_small(seed=0)
    b = sr.gae_small(seed=0)
    for k, v in a.arrays().items():
        np.testing.assert_array_equal(v, getattr(b, k))
    c = sr.gae_small(seed=1)
    assert not np.array_equal(a.reward, c.reward)
    assert not np.array_equal(a.reward, a.value)


def test_workload_shapes_and_rates():
    ro = sr.gae_trunc(N=512, T=1024)
    assert ro.reward.shape == (512, 1024) and ro.reward.dtype == np.float32
    assert ro.terminated.dtype == np.uint8 and ro.bootstrap.shape == (512,)
    assert abs(ro.terminated.mean() - 0.005) < 0.0005
    assert abs(ro.truncated.mean() - 0.002 * 0.995) < 0.0003
    assert not np.any(ro.terminated & ro.truncated)
    assert abs(ro.value.std() - 2.0) < 0.02
    ro = sr.vtrace(N=256, T=256)
    assert abs(ro.log_rho.std() - 0.5) < 0.01 and ro.truncated is None
    ro = sr.retrace(N=64, T=4096)
    assert np.all(ro.rho > 0) and abs(np.log(ro.rho).std() - 0.5) < 0.01
    assert abs(ro.terminated.mean() - 0.001) < 0.0004
