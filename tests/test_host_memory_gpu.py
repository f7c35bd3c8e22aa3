"""GPU parity with buffers in pinned host memory, which the kernels read and write in
place over NVLink-C2C: every estimator with all buffers on the host, inputs only, or
outputs only; the look-back path with host data and a device workspace; bf16 and fp16
inputs; the fused TD(lambda) call and the forward scans. Buffers the device cannot reach
(pageable host memory, a host workspace) are refused before anything is launched."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr
from parity_helpers import (ESTIMATORS, assert_parity, bf16_rounded, fp16_rounded, run_gpu,
                            run_oracle)

pytestmark = pytest.mark.gpu

MEMORY = -8  # RLCA_ERR_MEMORY


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()


@pytest.mark.parametrize("host", ["all", "inputs", "outputs"])
@pytest.mark.parametrize("N,T", [(37, 1024), (21, 777), (50, 128), (9, 3000)])
def test_every_estimator_in_host_memory(host, N, T):
    ro = sr.generic(N, T, seed=N * 7 + T, p_term=0.01, p_trunc=0.005)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, host=host), run_oracle(est, ro, {}),
                      f"{est} host={host} N={N} T={T}")


@pytest.mark.parametrize("ld_extra,offset", [(4, 0), (0, 2), (16, 4)])
def test_host_memory_layouts(ld_extra, offset):
    """128-bit and scalar access to host memory, and guard columns left untouched."""
    ro = sr.generic(11, 1024, seed=5 + ld_extra + offset)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, ld=1024 + ld_extra, offset=offset, host="all"),
                      run_oracle(est, ro, {}), f"{est} host ld+{ld_extra} off={offset}")


def test_gae_workload_from_host_memory():
    """The GAE workload's shape (which takes the bulk-copy kernel in device memory) with
    every buffer in pinned host memory."""
    ro = sr.gae_trunc(N=512, T=1024, seed=3)
    p = dict(gamma=ro.params["gamma"], lam=ro.params["lam"])
    assert_parity(run_gpu("gae", ro, p, host="all"), run_oracle("gae", ro, p), "gae host")


def test_lookback_with_host_data():
    ro = sr.generic(3, 5000, seed=8)
    ws = rlca.make_workspace(3, 5000)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, workspace=ws, host="all"), run_oracle(est, ro, {}),
                      f"{est} look-back host")
    assert rlca.workspace_check(ws) == 0


def test_bf16_inputs_in_host_memory():
    ro = bf16_rounded(sr.generic(16, 1024, seed=9))
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, in_dtype=torch.bfloat16, host="all"),
                      run_oracle(est, ro, {}), f"{est} bf16 host")


@pytest.mark.parametrize("T", [200, 1024, 1500])
def test_fp16_inputs_in_host_memory(T):
    """fp16 inputs in pinned host memory: the CTA tiles (the pipelined rows are for
    device memory) read them in place."""
    ro = fp16_rounded(sr.generic(16, T, seed=10 + T))
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, in_dtype=torch.float16, host="all"),
                      run_oracle(est, ro, {}), f"{est} fp16 host T={T}")


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def test_fused_td_and_forward_scans_in_host_memory():
    ro = sr.generic(24, 1100, seed=10)
    r, v, d, tr = _pinned(ro.reward), _pinned(ro.value), _pinned(ro.terminated), \
        _pinned(ro.truncated)
    tv, b = _pinned(ro.trunc_value), _pinned(ro.bootstrap)
    lams = (0.0, 0.9, 1.0)
    outs = rlca.rlca_td_lambda_multi(r, v, d, tr, tv, b, gamma=0.99, lams=lams)
    torch.cuda.synchronize()
    for lam, out in zip(lams, outs):
        assert not out.is_cuda and out.is_pinned()
        ref = oracle.td_lambda(ro.reward, ro.value, ro.terminated, ro.truncated,
                               ro.trunc_value, ro.bootstrap, gamma=0.99, lam=lam)
        assert_parity({"t": out.numpy().astype(np.float64)}, {"t": ref}, f"td multi {lam}")
    tr_out = rlca.rlca_eligibility_trace(v, d, tr, b, decay=0.9)
    ps_out = rlca.rlca_episodic_prefix_sum(v, d, tr, b)
    torch.cuda.synchronize()
    assert_parity({"e": tr_out.numpy().astype(np.float64)},
                  {"e": oracle.eligibility_trace(ro.value, ro.terminated, ro.truncated,
                                                 ro.bootstrap, decay=0.9)}, "trace host")
    assert_parity({"s": ps_out.numpy().astype(np.float64)},
                  {"s": oracle.episodic_prefix_sum(ro.value, ro.terminated, ro.truncated,
                                                   ro.bootstrap)}, "prefix sum host")


def test_pageable_host_memory_is_refused():
    """A pageable numpy buffer is not mapped for the device: the call returns
    RLCA_ERR_MEMORY and enqueues nothing (the output keeps its contents)."""
    N, T = 4, 64
    reward = np.ones((N, T), np.float32)
    term = torch.zeros((N, T), dtype=torch.uint8, device="cuda")
    out = torch.full((N, T), 7.0, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = rlca.lib().rlca_discounted_return(reward.ctypes.data, term.data_ptr(), None, None,
                                           None, 0.99, N, T, T, out.data_ptr(), st)
    assert rc == MEMORY
    assert b"pinned host memory" in rlca.lib().rlca_status_string(rc)
    pageable_out = np.empty((N, T), np.float32)
    ones = torch.ones((N, T), device="cuda")
    rc = rlca.lib().rlca_discounted_return(ones.data_ptr(), term.data_ptr(), None, None, None,
                                           0.99, N, T, T, pageable_out.ctypes.data, st)
    assert rc == MEMORY
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    with pytest.raises(ValueError, match="pinned"):
        rlca.rlca_discounted_return(torch.from_numpy(reward), term)


def test_host_workspace_is_refused():
    """The look-back state must be device memory: a pinned host workspace is refused
    and nothing is launched."""
    N, T = 2, 3000
    r = torch.randn((N, T), device="cuda")
    d = torch.zeros((N, T), dtype=torch.uint8, device="cuda")
    out = torch.full((N, T), 7.0, device="cuda")
    ws = torch.zeros(rlca.workspace_bytes(N, T), dtype=torch.uint8).pin_memory()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = rlca.lib().rlca_discounted_return_ex(r.data_ptr(), d.data_ptr(), None, None, None,
                                              0.99, N, T, T, out.data_ptr(), ws.data_ptr(),
                                              ws.numel(), st)
    assert rc == MEMORY
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
