"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics, not by the
oracle's own code.

- hand-computed golden examples (tests/golden/*.json), exact in binary floating point;
- closed-form discounted return for constant rewards;
- cross-estimator identities: GAE(lambda=1) = return - V, GAE(lambda=0) = TD error,
  TD(lambda) = GAE returns, on-policy V-trace = TD(lambda), on-policy Retrace with
  E_pi Q = Q and lambda = 1 telescopes to the discounted return;
- non-recursive sum definitions on tiny inputs (GAE sum of discounted TD errors,
  lambda-return as weighted n-step returns, IMPALA's V-trace sum, Munos et al.'s
  Retrace sum);
- episode-boundary semantics (rl-triton technical summary, Method section 3): every
  episode recomputed on its own gives bitwise the same values, and a NaN never leaves
  the episode it was planted in;
- row strides: padding columns are never read.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synthetic_rollouts as sr

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _arr(x, dt):
    return None if x is None else np.array(x, dtype=dt)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _case_inputs(c):
    g = {}
    for k in ("reward", "value", "trunc_value", "log_rho", "q_taken", "expected_q", "rho",
              "bootstrap", "bootstrap_ev"):
        g[k] = _arr(c.get(k), np.float32)
    for k in ("terminated", "truncated"):
        g[k] = _arr(c.get(k), np.uint8)
    return g


# ----------------------------------------------------------------------------- golden

def test_golden_discounted_return():
    for c in _load("discounted_return.json")["cases"]:
        g = _case_inputs(c)
        out = oracle.discounted_return(g["reward"], g["terminated"], g["truncated"],
                                       g["trunc_value"], g["bootstrap"], gamma=c["gamma"])
        np.testing.assert_array_equal(out, np.array(c["expected"]["returns"], float),
                                      err_msg=c["name"])


def test_golden_gae_and_td_lambda():
    for c in _load("gae_td_lambda.json")["cases"]:
        g = _case_inputs(c)
        adv, ret = oracle.gae(g["reward"], g["value"], g["terminated"], g["truncated"],
                              g["trunc_value"], g["bootstrap"], gamma=c["gamma"],
                              lam=c["lambda"])
        td = oracle.td_lambda(g["reward"], g["value"], g["terminated"], g["truncated"],
                              g["trunc_value"], g["bootstrap"], gamma=c["gamma"],
                              lam=c["lambda"])
        np.testing.assert_array_equal(adv, np.array(c["expected"]["advantages"], float))
        np.testing.assert_array_equal(ret, np.array(c["expected"]["returns"], float))
        np.testing.assert_array_equal(td, np.array(c["expected"]["td_lambda"], float))


def test_golden_vtrace():
    for c in _load("vtrace.json")["cases"]:
        g = _case_inputs(c)
        vs, pg = oracle.vtrace(g["reward"], g["value"], g["log_rho"], g["terminated"],
                               g["truncated"], g["trunc_value"], g["bootstrap"],
                               gamma=c["gamma"], lam=c["lambda"], rho_bar=c["rho_bar"],
                               c_bar=c["c_bar"], pg_rho_bar=c["pg_rho_bar"])
        np.testing.assert_array_equal(vs, np.array(c["expected"]["vs"], float), c["name"])
        np.testing.assert_array_equal(pg, np.array(c["expected"]["pg_advantages"], float),
                                      c["name"])


def test_golden_retrace():
    for c in _load("retrace.json")["cases"]:
        g = _case_inputs(c)
        q = oracle.retrace(g["reward"], g["q_taken"], g["expected_q"], g["rho"],
                           g["terminated"], g["truncated"], g["trunc_value"],
                           g["bootstrap_ev"], gamma=c["gamma"], lam=c["lambda"])
        np.testing.assert_array_equal(q, np.array(c["expected"]["q_ret"], float), c["name"])


# ------------------------------------------------------------------------ closed form

@pytest.mark.parametrize("gamma", [0.9, 0.5, 1.0, 0.0])
def test_closed_form_constant_reward(gamma):
    N, T, r, b = 2, 50, 0.75, -3.0
    reward = np.full((N, T), r, np.float32)
    term = np.zeros((N, T), np.uint8)
    boot = np.full((N,), b, np.float32)
    out = oracle.discounted_return(reward, term, bootstrap=boot, gamma=gamma)
    g = float(np.float32(gamma))
    for t in range(T):
        k = T - t
        if g == 1.0:
            want = r * k + b
        else:
            want = r * (1 - g ** k) / (1 - g) + g ** k * b
        np.testing.assert_allclose(out[:, t], want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- independent sum forms

def _episode_end(term, trunc, t, T):
    e = t
    while not (term[e] or (trunc is not None and trunc[e]) or e == T - 1):
        e += 1
    return e


def _end_value(term, trunc, tv, boot, e):
    """Value of the state after an episode's last step e (rl-triton Method section 3)."""
    if term[e]:
        return 0.0
    if trunc is not None and trunc[e]:
        return float(tv[e])
    return float(boot)


def _f(x):
    return float(np.float32(x))


def _small(seed, N=3, T=37, p_term=0.08, p_trunc=0.06):
    return sr.generic(N, T, seed=seed, p_term=p_term, p_trunc=p_trunc)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_discounted_return_sum_definition(seed):
    ro = _small(seed)
    gamma = 0.93
    out = oracle.discounted_return(ro.reward, ro.terminated, ro.truncated, ro.trunc_value,
                                   ro.bootstrap, gamma=gamma)
    g = _f(gamma)
    for n in range(ro.N):
        for t in range(ro.T):
            e = _episode_end(ro.terminated[n], ro.truncated[n], t, ro.T)
            want = sum(g ** (k - t) * float(ro.reward[n, k]) for k in range(t, e + 1))
            want += g ** (e - t + 1) * _end_value(ro.terminated[n], ro.truncated[n],
                                                  ro.trunc_value[n], ro.bootstrap[n], e)
            assert abs(out[n, t] - want) <= 1e-12 * (1 + abs(want))


@pytest.mark.parametrize("seed,lam", [(1, 0.9), (2, 0.0), (3, 1.0), (4, 0.37)])
def test_gae_sum_definition(seed, lam):
    """Schulman et al. 2016, eq. for GAE(gamma, lambda): A_t = sum_l (gamma lambda)^l
    delta_{t+l}, the sum running to the end of the episode inside the window."""
    ro = _small(seed)
    gamma = 0.95
    adv, ret = oracle.gae(ro.reward, ro.value, ro.terminated, ro.truncated, ro.trunc_value,
                          ro.bootstrap, gamma=gamma, lam=lam)
    g, l = _f(gamma), _f(lam)
    for n in range(ro.N):
        term, trunc = ro.terminated[n], ro.truncated[n]
        for t in range(ro.T):
            e = _episode_end(term, trunc, t, ro.T)
            want = 0.0
            for k in range(t, e + 1):
                nxt = float(ro.value[n, k + 1]) if k < e else _end_value(
                    term, trunc, ro.trunc_value[n], ro.bootstrap[n], e)
                delta = float(ro.reward[n, k]) + g * nxt - float(ro.value[n, k])
                want += (g * l) ** (k - t) * delta
            assert abs(adv[n, t] - want) <= 1e-12 * (1 + abs(want))
            assert ret[n, t] == adv[n, t] + float(ro.value[n, t])


@pytest.mark.parametrize("seed,lam", [(5, 0.8), (6, 0.0), (7, 1.0)])
def test_lambda_return_weighted_nstep_definition(seed, lam):
    """Sutton & Barto: the lambda-return is (1-lambda) sum_n lambda^(n-1) G^(n) with the
    remaining weight lambda^(m-1) on the full return to the episode end (m steps)."""
    ro = _small(seed)
    gamma = 0.9
    out = oracle.td_lambda(ro.reward, ro.value, ro.terminated, ro.truncated,
                           ro.trunc_value, ro.bootstrap, gamma=gamma, lam=lam)
    g, l = _f(gamma), _f(lam)
    for n in range(ro.N):
        term, trunc = ro.terminated[n], ro.truncated[n]
        for t in range(ro.T):
            e = _episode_end(term, trunc, t, ro.T)
            m = e - t + 1

            def nstep(k):
                s = sum(g ** j * float(ro.reward[n, t + j]) for j in range(k))
                tail = float(ro.value[n, t + k]) if k < m else _end_value(
                    term, trunc, ro.trunc_value[n], ro.bootstrap[n], e)
                return s + g ** k * tail

            want = (1 - l) * sum(l ** (k - 1) * nstep(k) for k in range(1, m)) \
                + l ** (m - 1) * nstep(m)
            assert abs(out[n, t] - want) <= 1e-11 * (1 + abs(want))


@pytest.mark.parametrize("seed,lam,rho_bar,c_bar,pg_bar",
                         [(8, 1.0, 1.0, 1.0, 1.0), (9, 0.9, 1.5, 0.8, 2.0),
                          (10, 1.0, 1e6, 1e6, 1e6)])
def test_vtrace_sum_definition(seed, lam, rho_bar, c_bar, pg_bar):
    """Espeholt et al. 2018, eq. (1): vs_s = V_s + sum_t gamma^(t-s) (prod_{i<t} c_i)
    rho_hat_t (r_t + gamma V_{t+1} - V_t); pg_s = rho_pg_s (r_s + gamma vs_{s+1} - V_s)."""
    ro = _small(seed)
    gamma = 0.97
    vs, pg = oracle.vtrace(ro.reward, ro.value, ro.log_rho, ro.terminated, ro.truncated,
                           ro.trunc_value, ro.bootstrap, gamma=gamma, lam=lam,
                           rho_bar=rho_bar, c_bar=c_bar, pg_rho_bar=pg_bar)
    g, l, rb, cb, pb = map(_f, (gamma, lam, rho_bar, c_bar, pg_bar))
    for n in range(ro.N):
        term, trunc = ro.terminated[n], ro.truncated[n]
        rho = [math.exp(float(x)) for x in ro.log_rho[n]]
        for s in range(ro.T):
            e = _episode_end(term, trunc, s, ro.T)
            endv = _end_value(term, trunc, ro.trunc_value[n], ro.bootstrap[n], e)
            want, prod = float(ro.value[n, s]), 1.0
            for t in range(s, e + 1):
                nxt = float(ro.value[n, t + 1]) if t < e else endv
                want += g ** (t - s) * prod * min(rb, rho[t]) * (
                    float(ro.reward[n, t]) + g * nxt - float(ro.value[n, t]))
                prod *= l * min(cb, rho[t])
            assert abs(vs[n, s] - want) <= 1e-11 * (1 + abs(want))
            q = vs[n, s + 1] if s < e else endv
            pg_want = min(pb, rho[s]) * (float(ro.reward[n, s]) + g * q - float(ro.value[n, s]))
            assert abs(pg[n, s] - pg_want) <= 1e-11 * (1 + abs(pg_want))


@pytest.mark.parametrize("seed,lam", [(11, 0.95), (12, 1.0), (13, 0.0)])
def test_retrace_sum_definition(seed, lam):
    """Munos et al. 2016: Q^ret_s = Q_s + sum_t gamma^(t-s) (c_{s+1} ... c_t)
    (r_t + gamma E_pi Q(s_{t+1},.) - Q_t), c = lambda min(1, rho)."""
    ro = _small(seed)
    gamma = 0.96
    out = oracle.retrace(ro.reward, ro.q_taken, ro.expected_q, ro.rho, ro.terminated,
                         ro.truncated, ro.trunc_value, ro.bootstrap, gamma=gamma, lam=lam)
    g, l = _f(gamma), _f(lam)
    for n in range(ro.N):
        term, trunc = ro.terminated[n], ro.truncated[n]
        for s in range(ro.T):
            e = _episode_end(term, trunc, s, ro.T)
            endv = _end_value(term, trunc, ro.trunc_value[n], ro.bootstrap[n], e)
            want, prod = float(ro.q_taken[n, s]), 1.0
            for t in range(s, e + 1):
                if t > s:
                    prod *= l * min(1.0, float(ro.rho[n, t]))
                nev = float(ro.expected_q[n, t + 1]) if t < e else endv
                want += g ** (t - s) * prod * (
                    float(ro.reward[n, t]) + g * nev - float(ro.q_taken[n, t]))
            assert abs(out[n, s] - want) <= 1e-11 * (1 + abs(want))


# ---------------------------------------------------------- cross-estimator identities

@pytest.mark.parametrize("seed", [0, 21])
def test_cross_estimator_identities(seed):
    ro = sr.generic(5, 200, seed=seed, p_term=0.03, p_trunc=0.02)
    gamma = 0.99
    args = (ro.terminated, ro.truncated, ro.trunc_value, ro.bootstrap)
    G = oracle.discounted_return(ro.reward, *args, gamma=gamma)
    v = ro.value.astype(np.float64)
    # GAE with lambda = 1 is the discounted return minus the value.
    adv1, _ = oracle.gae(ro.reward, ro.value, *args, gamma=gamma, lam=1.0)
    np.testing.assert_allclose(adv1, G - v, rtol=1e-11, atol=1e-11)
    # TD(lambda) with lambda = 1 is the discounted return.
    np.testing.assert_allclose(oracle.td_lambda(ro.reward, ro.value, *args, gamma=gamma,
                                                lam=1.0), G, rtol=1e-11, atol=1e-11)
    for lam in (0.0, 0.5, 0.95):
        adv, ret = oracle.gae(ro.reward, ro.value, *args, gamma=gamma, lam=lam)
        td = oracle.td_lambda(ro.reward, ro.value, *args, gamma=gamma, lam=lam)
        # TD(lambda) targets are the GAE returns.
        np.testing.assert_allclose(td, ret, rtol=1e-11, atol=1e-11)
        # On-policy V-trace (rho = 1, no clipping active) is TD(lambda).
        vs, _ = oracle.vtrace(ro.reward, ro.value, np.zeros_like(ro.reward), *args,
                              gamma=gamma, lam=lam)
        np.testing.assert_allclose(vs, td, rtol=1e-11, atol=1e-11)
    # GAE with lambda = 0 is the one-step TD error, and TD(0) = r + gamma * V(next).
    adv0, _ = oracle.gae(ro.reward, ro.value, *args, gamma=gamma, lam=0.0)
    td0 = oracle.td_lambda(ro.reward, ro.value, *args, gamma=gamma, lam=0.0)
    np.testing.assert_allclose(adv0, td0 - v, rtol=1e-11, atol=1e-11)
    # On-policy Retrace with E_pi Q = Q and lambda = 1 telescopes to the return.
    q = oracle.retrace(ro.reward, ro.value, ro.value, np.ones_like(ro.reward), *args,
                       gamma=gamma, lam=1.0)
    np.testing.assert_allclose(q, G, rtol=1e-10, atol=1e-10)
    # Retrace with lambda = 0 is the one-step expected-SARSA target, which for
    # E_pi Q = V is TD(0).
    q0 = oracle.retrace(ro.reward, ro.q_taken, ro.value, ro.rho, *args, gamma=gamma,
                        lam=0.0)
    np.testing.assert_allclose(q0, td0, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------- episode boundary semantics

def _all_estimators(ro, **kw):
    a = (ro.terminated, ro.truncated, ro.trunc_value, ro.bootstrap)
    out = {"dr": oracle.discounted_return(ro.reward, *a, gamma=0.97, **kw)}
    out["adv"], out["ret"] = oracle.gae(ro.reward, ro.value, *a, gamma=0.97, lam=0.9, **kw)
    out["td"] = oracle.td_lambda(ro.reward, ro.value, *a, gamma=0.97, lam=0.8, **kw)
    out["vs"], out["pg"] = oracle.vtrace(ro.reward, ro.value, ro.log_rho, *a, gamma=0.97,
                                         lam=0.9, rho_bar=1.2, c_bar=0.9, **kw)
    out["qret"] = oracle.retrace(ro.reward, ro.q_taken, ro.expected_q, ro.rho, *a,
                                 gamma=0.97, lam=0.95, **kw)
    return out


def _episodes(term, trunc, T):
    s = 0
    while s < T:
        e = _episode_end(term, trunc, s, T)
        yield s, e
        s = e + 1


def test_episode_split_is_bitwise_identical():
    """Each episode recomputed alone, ending terminal, truncated or at the window end
    with the same bootstrap, gives bitwise the same values: no credit crosses an
    episode boundary. A bootstrap that must not be read is NaN in the split problem."""
    ro = sr.generic(4, 300, seed=3, p_term=0.02, p_trunc=0.02)
    full = _all_estimators(ro)
    keys = ("reward", "terminated", "truncated", "trunc_value", "value", "log_rho",
            "q_taken", "expected_q", "rho")
    for n in range(ro.N):
        for s, e in _episodes(ro.terminated[n], ro.truncated[n], ro.T):
            sub = sr.Rollout(1, e - s + 1, reward=None, terminated=None)
            for k in keys:
                setattr(sub, k, np.ascontiguousarray(getattr(ro, k)[n:n + 1, s:e + 1]))
            window_end = e == ro.T - 1 and not ro.terminated[n, e] and not ro.truncated[n, e]
            sub.bootstrap = np.array([ro.bootstrap[n] if window_end else np.nan], np.float32)
            part = _all_estimators(sub)
            for k, v in full.items():
                np.testing.assert_array_equal(part[k][0], v[n, s:e + 1], err_msg=k)


@pytest.mark.parametrize("field", ["reward", "value", "q_taken", "expected_q", "rho",
                                   "log_rho"])
def test_nan_stays_in_its_episode(field):
    ro = sr.generic(3, 400, seed=4, p_term=0.02, p_trunc=0.01)
    clean = _all_estimators(ro)
    n, k = 1, 250
    getattr(ro, field)[n, k] = np.nan
    dirty = _all_estimators(ro)
    s = k
    while s > 0 and not (ro.terminated[n, s - 1] or ro.truncated[n, s - 1]):
        s -= 1
    for key in clean:
        a, b = clean[key].copy(), dirty[key].copy()
        a[n, s:k + 1] = 0.0
        b[n, s:k + 1] = 0.0
        np.testing.assert_array_equal(a, b, err_msg=f"{field} leaked into {key}")


def test_row_stride_padding_is_never_read():
    ro = sr.generic(3, 61, seed=5)
    base = _all_estimators(ro)
    ld = 64
    padded = sr.Rollout(ro.N, ro.T, reward=None, terminated=None)
    for k, v in ro.arrays().items():
        if v.ndim == 2:
            fill = 1 if v.dtype == np.uint8 else np.nan
            p = np.full((ro.N, ld), fill, v.dtype)
            p[:, :ro.T] = v
            setattr(padded, k, p)
        else:
            setattr(padded, k, v)
    strided = _all_estimators(padded, T=ro.T)
    for k in base:
        np.testing.assert_array_equal(base[k], strided[k], err_msg=k)
