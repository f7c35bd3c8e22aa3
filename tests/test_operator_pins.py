"""Pins on the scan formulation (no GPU): the pages' operator is associative, and any
bracketing of it over each estimator's (alpha_t, beta_t) pairs reproduces the fp64
oracle's textbook loops.

"rl-triton: High-Performance Triton GPU Kernels for Reinforcement Learning Credit
Assignment", Method section 1: every estimator is A_t = alpha_t + beta_t * A_{t+1},
solved as a scan over pairs with (aB, bB) (+) (aA, bA) = (aB + bB * aA, bA * bB), B the
earlier step. Method section 3: an episode's last step takes nothing from t+1 (a reset).
Here the reset is carried as a flag and the operator keeps the earlier element whole
when it resets. The pairs per estimator are the textbook ones (successor value sv_t at
an episode's last step: 0 if terminated, the truncation value if truncated, the per-env
bootstrap at the window end)."""
import random

import numpy as np
import pytest

import oracle
import synthetic_rollouts as sr


def combine(early, late):
    """(a, b, reset) of step range [early..late]: early applied after late."""
    a1, b1, r1 = early
    a2, b2, r2 = late
    if r1:
        return early
    return (a1 + b1 * a2, b1 * b2, r2)


def tree_fold(elems, lo, hi, rng):
    """Compose elems[lo:hi] with a random bracketing."""
    if hi - lo == 1:
        return elems[lo]
    mid = rng.randint(lo + 1, hi - 1)
    return combine(tree_fold(elems, lo, mid, rng), tree_fold(elems, mid, hi, rng))


def suffix_scan(elems, rng):
    """A_t = a of elems[t] (+) ... (+) elems[T-1], applied to A_T = 0."""
    return np.array([tree_fold(elems, t, len(elems), rng)[0] for t in range(len(elems))])


def test_operator_is_associative_with_resets():
    rng = np.random.default_rng(0)
    for _ in range(2000):
        x, y, z = [(float(rng.normal()), float(abs(rng.normal())), bool(rng.random() < 0.3))
                   for _ in range(3)]
        left = combine(combine(x, y), z)
        right = combine(x, combine(y, z))
        assert left[2] == right[2]
        assert abs(left[0] - right[0]) <= 1e-12 * (1 + abs(left[0]))
        assert abs(left[1] - right[1]) <= 1e-12 * (1 + abs(left[1]))


def _row(ro, n):
    T = ro.T
    term = ro.terminated[n].astype(bool)
    trunc = ro.truncated[n].astype(bool) & ~term
    end = np.zeros(T, bool)
    end[T - 1] = True
    stop = term | trunc | end
    sv = np.where(term, 0.0, np.where(trunc, ro.trunc_value[n].astype(np.float64),
                                      float(ro.bootstrap[n])))
    return term, trunc, stop, sv


def _f32(x):
    return float(np.float32(x))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bracketed_scans_match_the_oracle(seed):
    ro = sr.generic(3, 40, seed=seed, p_term=0.08, p_trunc=0.06)
    g, lam = _f32(0.97), _f32(0.9)  # fp32 parameters, widened; products in fp64
    gl = g * lam
    rng = random.Random(seed)
    ref_ret = oracle.discounted_return(ro.reward, ro.terminated, ro.truncated, ro.trunc_value,
                                       ro.bootstrap, gamma=g)
    ref_adv, _ = oracle.gae(ro.reward, ro.value, ro.terminated, ro.truncated, ro.trunc_value,
                            ro.bootstrap, gamma=g, lam=lam)
    ref_td = oracle.td_lambda(ro.reward, ro.value, ro.terminated, ro.truncated,
                              ro.trunc_value, ro.bootstrap, gamma=g, lam=lam)
    ref_q = oracle.retrace(ro.reward, ro.q_taken, ro.expected_q, ro.rho, ro.terminated,
                           ro.truncated, ro.trunc_value, ro.bootstrap, gamma=g, lam=lam)
    ref_vs, _ = oracle.vtrace(ro.reward, ro.value, ro.log_rho, ro.terminated, ro.truncated,
                              ro.trunc_value, ro.bootstrap, gamma=g, lam=1.0, rho_bar=1.0,
                              c_bar=1.0, pg_rho_bar=1.0)
    for n in range(ro.N):
        term, trunc, stop, sv = _row(ro, n)
        r = ro.reward[n].astype(np.float64)
        v = ro.value[n].astype(np.float64)
        v_next = np.append(v[1:], 0.0)
        nv = np.where(stop, sv, v_next)
        T = ro.T
        # discounted return: alpha = r + gamma * sv at an episode's last step, beta = gamma
        ret = [(r[t] + (g * sv[t] if stop[t] else 0.0), g, bool(stop[t])) for t in range(T)]
        np.testing.assert_allclose(suffix_scan(ret, rng), ref_ret[n], rtol=1e-12, atol=1e-12)
        # GAE: alpha = delta_t, beta = gamma * lambda
        adv = [(r[t] + g * nv[t] - v[t], gl, bool(stop[t])) for t in range(T)]
        np.testing.assert_allclose(suffix_scan(adv, rng), ref_adv[n], rtol=1e-12, atol=1e-12)
        # TD(lambda): alpha = r + gamma * (1 - lambda) * V_{t+1}, or r + gamma * sv at the end
        g1l = g * (1.0 - lam)
        td = [(r[t] + (g * sv[t] if stop[t] else g1l * v_next[t]), gl, bool(stop[t]))
              for t in range(T)]
        np.testing.assert_allclose(suffix_scan(td, rng), ref_td[n], rtol=1e-12, atol=1e-12)
        # Retrace: alpha = r + gamma * E_pi Q(s_{t+1}) - Q_t, beta = gamma * lambda *
        # min(1, rho_{t+1}); Q_ret = A + Q
        q = ro.q_taken[n].astype(np.float64)
        ev = ro.expected_q[n].astype(np.float64)
        rho = ro.rho[n].astype(np.float64)
        nev = np.where(stop, sv, np.append(ev[1:], 0.0))
        rho_next = np.append(rho[1:], 0.0)
        rt = [(r[t] + g * nev[t] - q[t], g * (lam * min(1.0, rho_next[t])), bool(stop[t]))
              for t in range(T)]
        np.testing.assert_allclose(suffix_scan(rt, rng) + q, ref_q[n], rtol=1e-11, atol=1e-11)
        # V-trace (lambda = 1, clips 1): alpha = min(1, rho_t) * delta_t, beta = gamma *
        # min(1, rho_t); vs = V + A
        rho_t = np.exp(ro.log_rho[n].astype(np.float64))
        vt = [(min(1.0, rho_t[t]) * (r[t] + g * nv[t] - v[t]), g * min(1.0, rho_t[t]),
               bool(stop[t])) for t in range(T)]
        np.testing.assert_allclose(suffix_scan(vt, rng) + v, ref_vs[n], rtol=1e-11, atol=1e-11)


def test_a_wrong_operand_order_is_caught():
    """Composing with the operands swapped (later applied after earlier) does not give
    the discounted return, so the order the kernels use is the one pinned above."""
    ro = sr.generic(1, 30, seed=4, p_term=0.0, p_trunc=0.0)
    g = _f32(0.9)
    r = ro.reward[0].astype(np.float64)
    T = ro.T
    elems = [(r[t] + (g * float(ro.bootstrap[0]) if t == T - 1 else 0.0), g, t == T - 1)
             for t in range(T)]
    right = elems[T - 1]
    wrong = (elems[T - 1][0], elems[T - 1][1], False)
    for t in range(T - 2, -1, -1):
        right = combine(elems[t], right)
        wrong = combine(wrong, elems[t])
    ref = oracle.discounted_return(ro.reward, ro.terminated, None, None, ro.bootstrap, gamma=g)
    assert abs(right[0] - ref[0, 0]) <= 1e-12 * (1 + abs(ref[0, 0]))
    assert abs(wrong[0] - ref[0, 0]) > 1e-6
