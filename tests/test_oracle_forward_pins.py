"""Pins for the oracle's forward-time scans (eligibility traces, episodic prefix sums):
hand-computed golden values, the closed form for constant inputs, the non-recursive
sum, numpy's cumsum per episode, the mirror identity with the (separately pinned)
discounted return on time-reversed inputs, per-episode recomputation and NaN isolation."""
import json
import os

import numpy as np
import pytest

import oracle
import synthetic_rollouts as sr

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f(x):
    return float(np.float32(x))


def test_golden_forward_scans():
    with open(os.path.join(GOLDEN, "forward_scans.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        x = np.array(c["x"], np.float32)
        d = np.array(c["terminated"], np.uint8)
        tr = np.array(c["truncated"], np.uint8) if "truncated" in c else None
        init = np.array(c["init"], np.float32) if "init" in c else None
        np.testing.assert_array_equal(
            oracle.eligibility_trace(x, d, tr, init, decay=c["decay"]),
            np.array(c["expected"]["trace"], float), c["name"])
        np.testing.assert_array_equal(oracle.episodic_prefix_sum(x, d, tr, init),
                                      np.array(c["expected"]["prefix_sum"], float), c["name"])


@pytest.mark.parametrize("decay", [0.9, 0.5, 1.0, 0.0])
def test_closed_form_constant_input(decay):
    N, T, x0, b = 2, 40, 0.25, -2.0
    x = np.full((N, T), x0, np.float32)
    d = np.zeros((N, T), np.uint8)
    init = np.full((N,), b, np.float32)
    out = oracle.eligibility_trace(x, d, init=init, decay=decay)
    g = _f(decay)
    for t in range(T):
        k = t + 1
        want = x0 * k + b if g == 1.0 else x0 * (1 - g ** k) / (1 - g) + g ** k * b
        np.testing.assert_allclose(out[:, t], want, rtol=1e-12, atol=1e-12)


def _starts(term, trunc, T):
    """Index of the first step of the episode each step belongs to (-1: the window's
    first episode, which also carries init)."""
    start, s = np.empty(T, int), -1
    for t in range(T):
        if t > 0 and (term[t - 1] or (trunc is not None and trunc[t - 1])):
            s = t
        start[t] = s
    return start


@pytest.mark.parametrize("seed,decay", [(1, 0.93), (2, 0.0), (3, 1.0)])
def test_sum_definition(seed, decay):
    ro = sr.generic(3, 45, seed=seed, p_term=0.08, p_trunc=0.05)
    out = oracle.eligibility_trace(ro.value, ro.terminated, ro.truncated, ro.bootstrap,
                                   decay=decay)
    g = _f(decay)
    for n in range(ro.N):
        st = _starts(ro.terminated[n], ro.truncated[n], ro.T)
        for t in range(ro.T):
            s = max(st[t], 0)
            want = sum(g ** (t - k) * float(ro.value[n, k]) for k in range(s, t + 1))
            if st[t] == -1:
                want += g ** (t + 1) * float(ro.bootstrap[n])
            assert abs(out[n, t] - want) <= 1e-12 * (1 + abs(want))


def test_prefix_sum_is_cumsum_per_episode():
    ro = sr.generic(4, 300, seed=4, p_term=0.03, p_trunc=0.02)
    out = oracle.episodic_prefix_sum(ro.value, ro.terminated, ro.truncated, ro.bootstrap)
    for n in range(ro.N):
        st = _starts(ro.terminated[n], ro.truncated[n], ro.T)
        for s in np.unique(st):
            idx = np.nonzero(st == s)[0]
            want = np.cumsum(ro.value[n, idx].astype(np.float64))
            if s == -1:
                want = want + float(ro.bootstrap[n])
            np.testing.assert_allclose(out[n, idx], want, rtol=1e-12, atol=1e-12)


def test_mirror_of_discounted_return():
    """Reversing time turns the forward trace into the backward discounted return: step
    t+1 starting an episode becomes a termination at the mirrored step, and init becomes
    the window-end bootstrap."""
    ro = sr.generic(5, 200, seed=5, p_term=0.02, p_trunc=0.02)
    decay = 0.97
    fwd = oracle.eligibility_trace(ro.value, ro.terminated, ro.truncated, ro.bootstrap,
                                   decay=decay)
    ended = (ro.terminated | ro.truncated).astype(np.uint8)
    x_rev = np.ascontiguousarray(ro.value[:, ::-1])
    term_rev = np.zeros_like(ended)
    term_rev[:, :-1] = ended[:, :-1][:, ::-1]  # ended[t-1] guards step t -> mirrored index
    back = oracle.discounted_return(x_rev, term_rev, bootstrap=ro.bootstrap, gamma=decay)
    np.testing.assert_allclose(fwd, back[:, ::-1], rtol=1e-12, atol=1e-12)


def test_episode_split_and_nan_isolation():
    ro = sr.generic(3, 250, seed=6, p_term=0.02, p_trunc=0.02)
    full = oracle.eligibility_trace(ro.value, ro.terminated, ro.truncated, ro.bootstrap,
                                    decay=0.9)
    for n in range(ro.N):
        st = _starts(ro.terminated[n], ro.truncated[n], ro.T)
        for s in np.unique(st):
            idx = np.nonzero(st == s)[0]
            init = np.array([ro.bootstrap[n] if s == -1 else 0.0], np.float32)
            part = oracle.eligibility_trace(np.ascontiguousarray(ro.value[n:n + 1, idx]),
                                            np.zeros((1, idx.size), np.uint8), init=init,
                                            decay=0.9)
            np.testing.assert_array_equal(part[0], full[n, idx])
    n, k = 1, 120
    ro.value[n, k] = np.nan
    dirty = oracle.eligibility_trace(ro.value, ro.terminated, ro.truncated, ro.bootstrap,
                                     decay=0.9)
    st = _starts(ro.terminated[n], ro.truncated[n], ro.T)
    e = k
    while e + 1 < ro.T and st[e + 1] == st[k]:
        e += 1
    a, b = full.copy(), dirty.copy()
    a[n, k:e + 1] = b[n, k:e + 1] = 0.0
    np.testing.assert_array_equal(a, b)
    assert np.isnan(dirty[n, k:e + 1]).all()
