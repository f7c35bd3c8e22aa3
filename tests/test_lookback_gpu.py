"""GPU parity of the look-back path (_ex entry points with a caller workspace, rows too
few to fill the GPU): every tile of every row runs in its own CTA and finds its
carry-in from the later tiles of its row. Same oracle and tolerance as the other parity
tests; the bounded wait is exercised by a testing entry point that makes every tile
withhold its state."""
import ctypes

import numpy as np
import pytest
import torch

import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr
from parity_helpers import ESTIMATORS, assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()


@pytest.mark.parametrize("N", [1, 3, 33])
@pytest.mark.parametrize("T", [1025, 2047, 2048, 2049, 4096, 4097, 10000])
def test_lookback_shape_grid(N, T):
    ro = sr.generic(N, T, seed=N * 131 + T, p_term=0.002, p_trunc=0.001)
    ws = rlca.make_workspace(N, T)
    assert ws is not None and ws.numel() == 256 + 32 * N * ((T + 1023) // 1024)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, workspace=ws), run_oracle(est, ro, {}),
                      f"{est} look-back N={N} T={T}")
    assert rlca.workspace_check(ws) == 0


def test_lookback_long_episodes_cross_many_tiles():
    """No terminations at all: every carry crosses every tile boundary of the row."""
    ro = sr.generic(4, 20000, seed=5, p_term=0.0, p_trunc=0.0)
    ro.truncated = None
    ws = rlca.make_workspace(4, 20000)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, dict(gamma=0.999, lam=0.999), workspace=ws),
                      run_oracle(est, ro, dict(gamma=0.999, lam=0.999)), f"{est} long")


def _epoch(ws):
    """Launches that used the workspace's look-back state (the header's first word)."""
    return int(ws[:4].cpu().view(torch.int32)[0])


def test_lookback_only_when_rows_cannot_fill_the_gpu():
    """With a workspace, look-back runs below two rows per SM and leaves the workspace
    untouched from there on (the row loop is faster once the rows fill the GPU)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = 2049
    for N, uses in ((2 * sms - 1, True), (2 * sms, False)):
        ro = sr.generic(N, T, seed=N, p_term=0.002, p_trunc=0.001)
        ws = rlca.make_workspace(N, T)
        ws.zero_()
        for i, est in enumerate(ESTIMATORS):
            assert_parity(run_gpu(est, ro, {}, workspace=ws), run_oracle(est, ro, {}),
                          f"{est} N={N} T={T}")
            assert _epoch(ws) == (i + 1 if uses else 0), (N, est)
        assert rlca.workspace_check(ws) == 0


@pytest.mark.parametrize("est", ["return", "gae"])
def test_very_long_rows(est):
    """Two rows of 2^20 + 7 steps (1025 tiles each, the last ragged): the look-back and
    the row loop over the whole row, with episodes that span hundreds of tiles."""
    N, T = 2, (1 << 20) + 7
    ro = sr.generic(N, T, seed=21, p_term=2e-6, p_trunc=1e-6)
    p = dict(gamma=0.999, lam=0.99)
    ref = run_oracle(est, ro, p)
    ws = rlca.make_workspace(N, T)
    assert_parity(run_gpu(est, ro, p, workspace=ws), ref, f"{est} look-back T={T}")
    assert _epoch(ws) == 1 and rlca.workspace_check(ws) == 0
    assert_parity(run_gpu(est, ro, p), ref, f"{est} row loop T={T}")


def test_ex_workload_retrace_2048x4096():
    """The retrace workload through the _ex call: 2048 rows fill the GPU, so the row
    loop runs and the workspace stays as it was, call after call."""
    ro = sr.retrace()
    p = dict(gamma=ro.params["gamma"], lam=ro.params["lam"])
    ws = rlca.make_workspace(ro.N, ro.T)
    ref = run_oracle("retrace", ro, p)
    for _ in range(3):
        assert_parity(run_gpu("retrace", ro, p, workspace=ws), ref, "retrace _ex")
    assert rlca.workspace_check(ws) == 0


def test_lookback_matches_row_loop_and_layouts():
    ro = sr.generic(5, 3000, seed=9)
    ws = rlca.make_workspace(5, 3000 + 4)
    for est in ESTIMATORS:
        for ld, off in ((3000, 0), (3004, 0), (3003, 1)):
            assert_parity(run_gpu(est, ro, {}, ld=ld, offset=off, workspace=ws),
                          run_oracle(est, ro, {}), f"{est} look-back ld={ld} off={off}")


def test_short_rows_ignore_the_workspace():
    assert rlca.workspace_bytes(100, 1024) == 0
    ro = sr.generic(7, 1024, seed=10)
    fake = torch.zeros(16, dtype=torch.uint8, device="cuda")  # unused when T <= 1024
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, workspace=fake), run_oracle(est, ro, {}), est)


def test_bounded_wait_reports_timeout_and_recovers():
    N, T = 8, 5000
    ro = sr.generic(N, T, seed=12, p_term=0.0, p_trunc=0.0)
    ws = rlca.make_workspace(N, T)
    r = torch.from_numpy(ro.reward).cuda()
    d = torch.from_numpy(ro.terminated).cuda()
    out = torch.empty_like(r)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = rlca.lib().rlca_testing_lookback_stall(r.data_ptr(), d.data_ptr(), N, T,
                                                out.data_ptr(), ws.data_ptr(), ws.numel(),
                                                64, st)
    assert rc == 0
    assert rlca.workspace_check(ws) == -7
    # Tiles that waited marked their outputs NaN; the row's last tile did not wait.
    host = out.cpu().numpy()
    waited = 1024 * ((T - 1) // 1024)  # every tile but the row's last
    assert np.isnan(host[:, :waited]).all() and np.isfinite(host[:, waited:]).all()
    assert rlca.workspace_check(ws) == 0  # the record was cleared
    # The workspace is ready for normal calls again.
    assert_parity(run_gpu("return", ro, {}, workspace=ws), run_oracle("return", ro, {}),
                  "after timeout")
    assert rlca.workspace_check(ws) == 0
