"""GPU parity: the CUDA path (through the C-ABI) against the fp64 oracle, element by
element, on the same seeded inputs. Tolerance: max|gpu - oracle| <= 1e-4 (1 + max|oracle|)
per output. Segmentation is checked exactly: a NaN planted in one episode leaves every
other value bitwise unchanged, and no write lands outside an output's [N, T] block."""
import copy

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
    return cuda_device


# ------------------------------------------------------------- the five workloads

def test_workload_gae_16x128():
    ro = sr.gae_small()
    p = dict(gamma=ro.params["gamma"], lam=ro.params["lam"])
    assert_parity(run_gpu("gae", ro, p), run_oracle("gae", ro, p), "gae 16x128")


def test_workload_return_td_4096x128():
    ro = sr.return_td()
    p = dict(gamma=ro.params["gamma"])
    assert_parity(run_gpu("return", ro, p), run_oracle("return", ro, p), "return 4096x128")
    for lam in ro.params["lams"]:
        p = dict(gamma=ro.params["gamma"], lam=lam)
        assert_parity(run_gpu("td_lambda", ro, p), run_oracle("td_lambda", ro, p),
                      f"td_lambda({lam}) 4096x128")


def test_workload_gae_trunc_4096x1024():
    ro = sr.gae_trunc()
    p = dict(gamma=ro.params["gamma"], lam=ro.params["lam"])
    assert_parity(run_gpu("gae", ro, p), run_oracle("gae", ro, p), "gae 4096x1024")


def test_workload_vtrace_8192x256():
    ro = sr.vtrace()
    p = {k: ro.params[k] for k in ("gamma", "lam", "rho_bar", "c_bar", "pg_rho_bar")}
    assert_parity(run_gpu("vtrace", ro, p), run_oracle("vtrace", ro, p), "vtrace 8192x256")


def test_workload_retrace_2048x4096():
    ro = sr.retrace()
    p = dict(gamma=ro.params["gamma"], lam=ro.params["lam"])
    assert_parity(run_gpu("retrace", ro, p), run_oracle("retrace", ro, p),
                  "retrace 2048x4096")


@pytest.mark.parametrize("est", ESTIMATORS)
def test_every_estimator_at_4096x1024(est):
    """The roofline shape, for every estimator, with truncation present."""
    ro = sr.generic(4096, 1024, seed=7, p_term=0.005, p_trunc=0.002)
    assert_parity(run_gpu(est, ro, {}), run_oracle(est, ro, {}), f"{est} 4096x1024")


# -------------------------------------------------------------------- edge grid

T_GRID = [1, 2, 3, 4, 5, 15, 16, 17, 31, 127, 128, 129, 255, 256, 257, 511, 512, 513,
          1023, 1024, 1025, 2047, 2048, 2049, 4095, 4096, 4097]


@pytest.mark.parametrize("N", [1, 3, 33])
@pytest.mark.parametrize("T", T_GRID)
def test_shape_grid(N, T):
    ro = sr.generic(N, T, seed=N * 10007 + T, p_term=0.03, p_trunc=0.02)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}), run_oracle(est, ro, {}), f"{est} N={N} T={T}")


def _pattern(ro, name):
    N, T = ro.N, ro.T
    term = np.zeros((N, T), np.uint8)
    trunc = np.zeros((N, T), np.uint8)
    if name == "all_done":
        term[:] = 1
    elif name == "all_truncated":
        trunc[:] = 1
    elif name == "done_at_0":
        term[:, 0] = 1
    elif name == "done_at_last":
        term[:, -1] = 1
    elif name == "trunc_at_last":
        trunc[:, -1] = 1
    elif name == "done_and_trunc_same_step":
        term[:, T // 2] = 1
        trunc[:, T // 2] = 1
        trunc[:, T // 3] = 1
    elif name == "alternating":
        term[:, ::2] = 1
        trunc[:, 1::4] = 1
    ro.terminated, ro.truncated = term, trunc
    return ro


@pytest.mark.parametrize("pattern", ["no_done", "all_done", "all_truncated", "done_at_0",
                                     "done_at_last", "trunc_at_last",
                                     "done_and_trunc_same_step", "alternating"])
@pytest.mark.parametrize("T", [1, 7, 1024, 1500, 4100])
def test_flag_patterns(pattern, T):
    ro = _pattern(sr.generic(5, T, seed=T), pattern)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}), run_oracle(est, ro, {}), f"{est} {pattern} T={T}")


def test_no_truncation_and_no_bootstrap():
    ro = sr.generic(9, 700, seed=11)
    ro.truncated = None
    ro.trunc_value = None
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}), run_oracle(est, ro, {}), f"{est} no trunc")
    ro.bootstrap = None
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}), run_oracle(est, ro, {}), f"{est} no bootstrap")


@pytest.mark.parametrize("params", [dict(gamma=0.0), dict(gamma=1.0), dict(lam=0.0),
                                    dict(lam=1.0), dict(gamma=1.0, lam=1.0),
                                    dict(gamma=0.0, lam=0.0)])
def test_parameter_extremes(params):
    ro = sr.generic(7, 1100, seed=12, p_term=0.01, p_trunc=0.01)
    for est in ESTIMATORS:
        p = {k: v for k, v in params.items() if est != "return" or k == "gamma"}
        assert_parity(run_gpu(est, ro, p), run_oracle(est, ro, p), f"{est} {params}")


def test_importance_ratio_extremes():
    ro = sr.generic(6, 900, seed=13)
    ro.log_rho = np.where(np.arange(900)[None, :] % 3 == 0, 20.0, -20.0).astype(np.float32) \
        * np.ones((6, 1), np.float32)
    ro.rho = np.exp(ro.log_rho.astype(np.float64)).astype(np.float32)
    for p in (dict(rho_bar=1.0, c_bar=1.0), dict(rho_bar=5.0, c_bar=0.5, pg_rho_bar=2.0),
              dict(rho_bar=1e30, c_bar=1e30, pg_rho_bar=1e30, gamma=0.9)):
        assert_parity(run_gpu("vtrace", ro, p), run_oracle("vtrace", ro, p), f"vtrace {p}")
    for lam in (0.0, 0.5, 1.0):
        p = dict(lam=lam)
        assert_parity(run_gpu("retrace", ro, p), run_oracle("retrace", ro, p),
                      f"retrace lam={lam}")


@pytest.mark.parametrize("T", [300, 1024, 3000])
def test_retrace_zero_ratio_inside_episodes(T):
    """rho = +0 is inside Retrace's domain: c_{t+1} = 0 cuts the trace as the formula
    does (beta_t = +0, not a reset). Planted inside long episodes, at chunk and tile
    boundaries, then with a NaN later in the episode (0 * NaN is NaN on both sides), and
    on the look-back path for rows longer than a tile."""
    ro = sr.generic(4, T, seed=71 + T, p_term=0.0005, p_trunc=0.0)
    zeros = [t for t in (5, 255, 256, 257, 700, 1023, 1024, 2047, 2048, 2900) if t < T]
    ro.rho = ro.rho.copy()
    for i, t in enumerate(zeros):
        ro.rho[i % 4, t] = 0.0
        ro.rho[(i + 1) % 4, t] = 0.0
    assert not np.signbit(ro.rho).any()
    for lam in (0.95, 1.0):
        p = dict(lam=lam)
        assert_parity(run_gpu("retrace", ro, p), run_oracle("retrace", ro, p),
                      f"retrace rho=+0 lam={lam}")
    ro.reward = ro.reward.copy()
    ro.reward[1, min(T - 1, zeros[1] + 10)] = np.nan
    ro.reward[2, min(T - 1, zeros[-1] + 3)] = np.nan
    ref = run_oracle("retrace", ro, {})
    assert np.isnan(ref["q_ret"][1, :zeros[1]]).any()  # the NaN crosses the zero ratio
    assert_parity(run_gpu("retrace", ro, {}), ref, "retrace rho=+0 with NaN")
    if T > 1024:
        ws = rlca.make_workspace(ro.N, T, "cuda")
        assert_parity(run_gpu("retrace", ro, {}, workspace=ws), ref,
                      "retrace rho=+0 with NaN, look-back")


def test_retrace_negative_ratio_ends_the_trace():
    """Outside the domain (rho < 0 or -0.0) a ratio is read as the end of the trace: with
    finite values the result equals the formula with that ratio replaced by +0."""
    ro = sr.generic(3, 1500, seed=77, p_term=0.001, p_trunc=0.0)
    neg = ro.rho.copy()
    neg[0, 100] = -0.0
    neg[1, 600] = -0.5
    neg[2, 1024] = -3.0
    neg[0, 1400] = -0.0
    clamped = ro.rho.copy()
    clamped[neg <= 0] = 0.0
    ro_neg, ro_ref = copy.copy(ro), copy.copy(ro)
    ro_neg.rho, ro_ref.rho = neg, clamped
    assert_parity(run_gpu("retrace", ro_neg, {}), run_oracle("retrace", ro_ref, {}),
                  "retrace negative rho")


@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (4, 0), (3, 0), (0, 1), (1, 3), (8, 4)])
@pytest.mark.parametrize("T", [5, 128, 1030, 3000])
def test_row_stride_and_alignment(ld_extra, offset, T):
    """ld > T and bases that are not 16-byte aligned take the scalar path; no write may
    land in the padding columns or outside the block."""
    ro = sr.generic(4, T, seed=14 + T)
    for est in ESTIMATORS:
        g = run_gpu(est, ro, {}, ld=T + ld_extra, offset=offset)
        assert_parity(g, run_oracle(est, ro, {}), f"{est} ld=T+{ld_extra} off={offset}")


@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (4, 0), (3, 0), (0, 1)])
@pytest.mark.parametrize("T", [257, 300, 512, 513, 777, 1023, 1024])
def test_without_truncation(ld_extra, offset, T):
    """No truncation tensor at all: GAE rows longer than half a tile then take the CTA
    kernel (one row per CTA) instead of the pipelined warp-owned rows."""
    ro = sr.generic(37, T, seed=90 + T, p_term=0.01, p_trunc=0.0)
    ro.truncated = None
    for est in ESTIMATORS:
        g = run_gpu(est, ro, {}, ld=T + ld_extra, offset=offset)
        assert_parity(g, run_oracle(est, ro, {}), f"{est} no truncation T={T} "
                      f"ld=T+{ld_extra} off={offset}")


@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (16, 0), (16, 4), (8, 2), (4, 0)])
@pytest.mark.parametrize("T", [256, 1024, 2048])
def test_access_widths(ld_extra, offset, T):
    """Each access width on the same inputs: 256-bit (32-byte aligned rows: ld % 8 == 0,
    offset 0), 128-bit (offset 4 floats or ld % 8 == 4), scalar (offset 2). GAE with
    truncation at T = 1024 takes the pipelined warp-owned rows at both aligned levels."""
    ro = sr.generic(29, T, seed=70 + T + ld_extra + offset, p_term=0.01, p_trunc=0.005)
    for est in ESTIMATORS:
        g = run_gpu(est, ro, {}, ld=T + ld_extra, offset=offset)
        assert_parity(g, run_oracle(est, ro, {}), f"{est} T={T} ld=T+{ld_extra} off={offset}")


@pytest.mark.parametrize("T", [13, 250, 517, 1001, 1023, 3001])
def test_wide_access_with_ragged_tails(T):
    """Rows padded to a multiple of 8 floats (256-bit access) whose length is not: every
    thread but the row's last moves its steps with wide accesses, the last one steps
    through its tail with scalar ones."""
    ld = (T + 7) // 8 * 8
    ro = sr.generic(19, T, seed=T + 5, p_term=0.01, p_trunc=0.005)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, ld=ld), run_oracle(est, ro, {}),
                      f"{est} T={T} ld={ld}")


def test_bool_flags():
    ro = sr.generic(8, 333, seed=15, p_term=0.05, p_trunc=0.05)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, bool_flags=True), run_oracle(est, ro, {}),
                      f"{est} bool flags")


def test_optional_second_output():
    ro = sr.generic(3, 1500, seed=16)
    for est in ("gae", "vtrace"):
        g = run_gpu(est, ro, {}, drop_second_output=True)
        assert len(g) == 1
        assert_parity(g, run_oracle(est, ro, {}), f"{est} single output")


# ------------------------------------------------------------- exact segmentation

@pytest.mark.parametrize("T", [300, 2600])
@pytest.mark.parametrize("field", ["reward", "value", "q_taken", "expected_q", "rho",
                                   "log_rho", "trunc_value"])
def test_nan_stays_in_its_episode(field, T):
    ro = sr.generic(3, T, seed=17, p_term=0.01, p_trunc=0.01)
    n, k = 1, T * 2 // 3
    if field == "trunc_value":
        ro.terminated[n, k] = 0
        ro.truncated[n, k] = 1
    clean = {e: run_gpu(e, ro, {}) for e in ESTIMATORS}
    getattr(ro, field)[n, k] = np.nan
    s = k
    while s > 0 and not (ro.terminated[n, s - 1] or ro.truncated[n, s - 1]):
        s -= 1
    for est in ESTIMATORS:
        dirty = run_gpu(est, ro, {})
        for name, a in clean[est].items():
            a, b = a.copy(), dirty[name].copy()
            a[n, s:k + 1] = 0.0
            b[n, s:k + 1] = 0.0
            assert np.array_equal(a, b), f"NaN in {field} leaked into {est}/{name}"


def test_repeatable():
    ro = sr.generic(64, 2000, seed=18)
    for est in ESTIMATORS:
        a, b = run_gpu(est, ro, {}), run_gpu(est, ro, {})
        for name in a:
            assert np.array_equal(a[name], b[name]), est


def test_empty_problems():
    import segmented_associative_scan_gb300 as rlca
    dev = "cuda:0"
    for N, T in ((0, 16), (4, 0), (0, 0)):
        r = torch.zeros((N, T), device=dev)
        d = torch.zeros((N, T), dtype=torch.uint8, device=dev)
        assert rlca.rlca_discounted_return(r, d).shape == (N, T)
        adv, ret = rlca.rlca_gae(r, r, d)
        assert adv.shape == (N, T) and ret.shape == (N, T)
    torch.cuda.synchronize()


def test_flag_bytes_any_nonzero_value_is_set():
    """Flags are bytes with 0 = clear and any nonzero value = set (0x80, 0xff, 7, ...)."""
    ro = sr.generic(6, 2100, seed=19, p_term=0.03, p_trunc=0.03)
    rng = np.random.default_rng(3)
    for name in ("terminated", "truncated"):
        f = getattr(ro, name)
        vals = rng.choice(np.array([1, 2, 7, 0x10, 0x7f, 0x80, 0x81, 0xfe, 0xff], np.uint8),
                          size=f.shape)
        setattr(ro, name, np.where(f != 0, vals, 0).astype(np.uint8))
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}), run_oracle(est, ro, {}), f"{est} flag bytes")
        assert_parity(run_gpu(est, ro, {}, ld=2104, offset=0), run_oracle(est, ro, {}),
                      f"{est} flag bytes, padded rows")
