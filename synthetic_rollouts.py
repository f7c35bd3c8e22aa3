"""Seeded synthetic rollouts shaped like the workloads of "rl-triton: High-Performance
Triton GPU Kernels for Reinforcement Learning Credit Assignment" (Problem statement:
[num_envs, seq_len] reward/value/done tensors; Results: e.g. 4,096 envs x 128 steps).

This module only draws random numbers. It holds none of the estimators' arithmetic, so
both the fp64 oracle and the CUDA path can take their inputs from it.

Every tensor comes from its own numpy PCG64 substream, derived from (seed, tensor name),
so adding a tensor never changes the others. Arrays are host numpy arrays:
float32 [N, T] data, uint8 [N, T] flags (0/1), float32 [N] bootstrap values.

"N(mu, s)" in the workload descriptions means mean mu and standard deviation s.
Truncation is drawn only where the step is not terminated, so both rates stay as stated.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field

import numpy as np

_SUBSTREAM = {
    "reward": 1, "spike": 2, "value": 3, "bootstrap": 4, "terminated": 5,
    "truncated": 6, "trunc_value": 7, "log_rho": 8, "q_taken": 9, "expected_q": 10,
    "rho": 11, "bootstrap_ev": 12,
}


def _rng(seed: int, name: str) -> np.random.Generator:
    key = _SUBSTREAM.get(name)
    if key is None:
        key = 1000 + zlib.crc32(name.encode())
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), key])))


def normal(seed, name, shape, std=1.0):
    return (_rng(seed, name).standard_normal(shape) * std).astype(np.float32)


def bernoulli(seed, name, shape, p):
    return (_rng(seed, name).random(shape) < p).astype(np.uint8)


@dataclass
class Rollout:
    """One synthetic batch. Fields that an estimator does not use are None."""
    N: int
    T: int
    reward: np.ndarray
    terminated: np.ndarray
    truncated: np.ndarray | None = None
    trunc_value: np.ndarray | None = None
    bootstrap: np.ndarray | None = None
    value: np.ndarray | None = None
    log_rho: np.ndarray | None = None
    q_taken: np.ndarray | None = None
    expected_q: np.ndarray | None = None
    rho: np.ndarray | None = None
    params: dict = field(default_factory=dict)

    def arrays(self) -> dict:
        return {k: v for k, v in self.__dict__.items() if isinstance(v, np.ndarray)}

    def nbytes(self) -> int:
        return sum(v.nbytes for v in self.arrays().values())


def _flags(seed, N, T, p_term, p_trunc):
    term = bernoulli(seed, "terminated", (N, T), p_term)
    trunc = None
    if p_trunc:
        trunc = bernoulli(seed, "truncated", (N, T), p_trunc) & (1 - term)
    return term, trunc


def gae_small(N=16, T=128, seed=0):
    """GAE, fp32, [16,128]: r,V ~ N(0,1), one bootstrap value per env ~ N(0,1),
    dones ~ B(0.01), truncations ~ B(0.005) with next-state values ~ N(0,1),
    gamma=0.99, lambda=0.95."""
    term, trunc = _flags(seed, N, T, 0.01, 0.005)
    return Rollout(N, T, reward=normal(seed, "reward", (N, T)), terminated=term,
                   truncated=trunc, trunc_value=normal(seed, "trunc_value", (N, T)),
                   bootstrap=normal(seed, "bootstrap", (N,)),
                   value=normal(seed, "value", (N, T)),
                   params=dict(gamma=0.99, lam=0.95))


def return_td(N=4096, T=128, seed=0):
    """Discounted return and TD(lambda), fp32, [4096,128]: r,V ~ N(0,1), bootstrap ~ N(0,1),
    dones ~ B(0.02), no truncation, gamma=0.99, lambda in {0, 0.9, 1.0}."""
    term, _ = _flags(seed, N, T, 0.02, 0.0)
    return Rollout(N, T, reward=normal(seed, "reward", (N, T)), terminated=term,
                   bootstrap=normal(seed, "bootstrap", (N,)),
                   value=normal(seed, "value", (N, T)),
                   params=dict(gamma=0.99, lams=(0.0, 0.9, 1.0)))


def gae_trunc(N=4096, T=1024, seed=0):
    """GAE with truncation bootstrapping, fp32, [4096,1024]: r ~ N(0,1) plus +10 spikes
    (p=0.001), V ~ N(0,2), bootstrap ~ N(0,2), dones ~ B(0.005), truncations ~ B(0.002)
    each with a next-state value ~ N(0,2), gamma=0.995, lambda=0.95."""
    term, trunc = _flags(seed, N, T, 0.005, 0.002)
    spikes = bernoulli(seed, "spike", (N, T), 0.001).astype(np.float32) * np.float32(10.0)
    return Rollout(N, T, reward=normal(seed, "reward", (N, T)) + spikes, terminated=term,
                   truncated=trunc, trunc_value=normal(seed, "trunc_value", (N, T), 2.0),
                   bootstrap=normal(seed, "bootstrap", (N,), 2.0),
                   value=normal(seed, "value", (N, T), 2.0),
                   params=dict(gamma=0.995, lam=0.95))


def vtrace(N=8192, T=256, seed=0):
    """V-trace, fp32, [8192,256]: r,V ~ N(0,1), log ratios ~ N(0,0.5), rho_bar=c_bar=1,
    dones ~ B(0.01), gamma=0.99, bootstrap ~ N(0,1)."""
    term, _ = _flags(seed, N, T, 0.01, 0.0)
    return Rollout(N, T, reward=normal(seed, "reward", (N, T)), terminated=term,
                   bootstrap=normal(seed, "bootstrap", (N,)),
                   value=normal(seed, "value", (N, T)),
                   log_rho=normal(seed, "log_rho", (N, T), 0.5),
                   params=dict(gamma=0.99, lam=1.0, rho_bar=1.0, c_bar=1.0, pg_rho_bar=1.0))


def retrace(N=2048, T=4096, seed=0):
    """Retrace, fp32, [2048,4096]: r, Q(s,a), E_pi Q(s,.) ~ N(0,1) independent,
    rho = exp(N(0,0.5)), lambda=0.95, gamma=0.99, dones ~ B(0.001),
    bootstrap E_pi Q ~ N(0,1)."""
    term, _ = _flags(seed, N, T, 0.001, 0.0)
    rho = np.exp(normal(seed, "rho", (N, T), 0.5).astype(np.float64)).astype(np.float32)
    return Rollout(N, T, reward=normal(seed, "reward", (N, T)), terminated=term,
                   bootstrap=normal(seed, "bootstrap_ev", (N,)),
                   q_taken=normal(seed, "q_taken", (N, T)),
                   expected_q=normal(seed, "expected_q", (N, T)),
                   rho=rho, params=dict(gamma=0.99, lam=0.95))


def traces(N=4096, T=1024, seed=0):
    """Forward scans (eligibility traces, episodic prefix sums), fp32: per-step inputs
    x ~ N(0,1) (in `value`), dones ~ B(0.01), truncations ~ B(0.005), carried-in values
    ~ N(0,1) (in `bootstrap`), decay = gamma * lambda = 0.99 * 0.95."""
    term, trunc = _flags(seed, N, T, 0.01, 0.005)
    return Rollout(N, T, reward=normal(seed, "reward", (N, T)), terminated=term,
                   truncated=trunc, bootstrap=normal(seed, "bootstrap", (N,)),
                   value=normal(seed, "value", (N, T)),
                   params=dict(gamma=0.99, lam=0.95, decay=0.99 * 0.95))


# The five workloads, by name, with their full sizes.
WORKLOADS = {
    "gae_16x128": (gae_small, dict(N=16, T=128)),
    "return_td_4096x128": (return_td, dict(N=4096, T=128)),
    "gae_trunc_4096x1024": (gae_trunc, dict(N=4096, T=1024)),
    "vtrace_8192x256": (vtrace, dict(N=8192, T=256)),
    "retrace_2048x4096": (retrace, dict(N=2048, T=4096)),
}


def generic(N, T, seed=0, p_term=0.01, p_trunc=0.005, std=1.0):
    """Every input any estimator takes, for edge-case grids: all data ~ N(0,std),
    log ratios ~ N(0,0.5), rho = exp(log ratios)."""
    term, trunc = _flags(seed, N, T, p_term, p_trunc)
    log_rho = normal(seed, "log_rho", (N, T), 0.5)
    return Rollout(N, T, reward=normal(seed, "reward", (N, T), std), terminated=term,
                   truncated=trunc, trunc_value=normal(seed, "trunc_value", (N, T), std),
                   bootstrap=normal(seed, "bootstrap", (N,), std),
                   value=normal(seed, "value", (N, T), std), log_rho=log_rho,
                   q_taken=normal(seed, "q_taken", (N, T), std),
                   expected_q=normal(seed, "expected_q", (N, T), std),
                   rho=np.exp(log_rho.astype(np.float64)).astype(np.float32))
