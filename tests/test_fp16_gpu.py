"""GPU parity of the fp16-input entry points (_fp16): every per-step data input is
rounded to fp16 first, the kernels widen each value to fp32 exactly (CUDA's conversion)
and compute in fp32, and the result is compared with the fp64 oracle on the same widened
values, with the tolerance of the fp32 paths. Covers warp-owned rows, the pipelined warp
rows, CTA tiles, the row loop, the forward scans, strided and unaligned layouts, and the
ends of the fp16 range: subnormals (down to 2^-24) and +-65504."""
import numpy as np
import pytest
import torch

import oracle
import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr
from parity_helpers import ESTIMATORS, assert_parity, fp16_rounded, run_gpu, run_oracle

pytestmark = pytest.mark.gpu
HF = torch.float16


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()


@pytest.mark.parametrize("T", [1, 7, 128, 256, 300, 520, 1024, 1100, 4096])
def test_fp16_reverse_estimators(T):
    ro = fp16_rounded(sr.generic(9, T, seed=600 + T, p_term=0.02, p_trunc=0.01))
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, in_dtype=HF), run_oracle(est, ro, {}),
                      f"{est} fp16 T={T}")


def _plant_extremes(ro, seed):
    """Subnormal, smallest-normal and largest finite fp16 values planted in every data
    input (ratios kept >= 0, log-ratios small enough that exp stays finite)."""
    rng = np.random.default_rng(seed)
    special = np.array([2.0 ** -24, -2.0 ** -24, 3 * 2.0 ** -20, -1023 * 2.0 ** -24,
                        2.0 ** -14, 65504.0, -65504.0, 0.0, -0.0], np.float32)
    for k in ("reward", "value", "trunc_value", "q_taken", "expected_q", "log_rho", "rho"):
        a = getattr(ro, k).copy()
        mask = rng.random(a.shape) < 0.05
        vals = special[rng.integers(0, len(special), a.shape)]
        if k == "log_rho":
            vals = np.clip(vals, -30.0, 30.0)
        if k == "rho":
            vals = np.abs(vals)
        a[mask] = vals[mask]
        setattr(ro, k, a)
    return fp16_rounded(ro)


@pytest.mark.parametrize("T", [100, 700, 1024, 2500])
def test_fp16_range_ends(T):
    ro = _plant_extremes(sr.generic(8, T, seed=700 + T, p_term=0.02, p_trunc=0.01), T)
    sub = np.abs(ro.reward[(ro.reward != 0) & (np.abs(ro.reward) < 2.0 ** -14)])
    assert sub.size and sub.min() == 2.0 ** -24  # subnormals reach the kernels unchanged
    assert np.abs(ro.value).max() == 65504.0
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, in_dtype=HF), run_oracle(est, ro, {}),
                      f"{est} fp16 extremes T={T}")


@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (8, 0), (4, 0), (0, 2), (3, 1), (16, 8)])
@pytest.mark.parametrize("T", [200, 1000, 1024])
def test_fp16_layouts(T, ld_extra, offset):
    """ld % 8 == 0 with aligned bases takes 128-bit loads (and the pipelined warp rows on
    rows of 257-1024 steps); the rest the scalar path."""
    ro = fp16_rounded(sr.generic(5, T, seed=800 + T + ld_extra, p_term=0.01, p_trunc=0.01))
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, ld=T + ld_extra, offset=offset, in_dtype=HF),
                      run_oracle(est, ro, {}), f"{est} fp16 T={T} ld+{ld_extra} off={offset}")


@pytest.mark.parametrize("trunc", [True, False])
@pytest.mark.parametrize("T", [257, 263, 512, 513, 768, 1016, 1024])
def test_fp16_pipelined_rows(T, trunc):
    ro = fp16_rounded(sr.generic(21, T, seed=900 + T, p_term=0.01,
                                 p_trunc=0.01 if trunc else 0.0))
    if not trunc:
        ro.truncated = None
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, in_dtype=HF), run_oracle(est, ro, {}),
                      f"{est} fp16 T={T} trunc={trunc}")


def test_fp16_workloads():
    for est, ro, p in (("gae", sr.gae_trunc(), dict(gamma=0.995, lam=0.95)),
                       ("vtrace", sr.vtrace(), dict(gamma=0.99, lam=1.0)),
                       ("retrace", sr.retrace(N=512), dict(gamma=0.99, lam=0.95))):
        ro = fp16_rounded(ro)
        assert_parity(run_gpu(est, ro, p, in_dtype=HF), run_oracle(est, ro, p), f"{est} fp16")


@pytest.mark.parametrize("T", [5, 200, 1024, 3000])
def test_fp16_forward_scans(T):
    ro = fp16_rounded(sr.generic(6, T, seed=950 + T, p_term=0.02, p_trunc=0.01))
    dev = "cuda:0"
    x = torch.from_numpy(ro.value).to(dev).to(HF)
    d = torch.from_numpy(ro.terminated).to(dev)
    tr = torch.from_numpy(ro.truncated).to(dev)
    init = torch.from_numpy(ro.bootstrap).to(dev)
    got = rlca.rlca_eligibility_trace(x, d, tr, init, decay=0.9)
    ref = oracle.eligibility_trace(ro.value, ro.terminated, ro.truncated, ro.bootstrap, decay=0.9)
    assert_parity({"o": got.cpu().numpy().astype(np.float64)}, {"o": ref}, f"trace T={T}")
    got = rlca.rlca_episodic_prefix_sum(x, d, tr, init)
    ref = oracle.episodic_prefix_sum(ro.value, ro.terminated, ro.truncated, ro.bootstrap)
    assert_parity({"o": got.cpu().numpy().astype(np.float64)}, {"o": ref}, f"sum T={T}")


def test_fp16_rejects_mixed_dtypes_and_workspace():
    dev = "cuda:0"
    r = torch.zeros((4, 2048), device=dev, dtype=HF)
    d = torch.zeros((4, 2048), device=dev, dtype=torch.uint8)
    with pytest.raises(TypeError):
        rlca.rlca_gae(r, torch.zeros((4, 2048), device=dev, dtype=torch.bfloat16), d)
    with pytest.raises(TypeError):
        rlca.rlca_gae(r, torch.zeros((4, 2048), device=dev, dtype=torch.float32), d)
    with pytest.raises(ValueError):
        rlca.rlca_gae(r, r, d, workspace=torch.zeros(4096, dtype=torch.uint8, device=dev))


def test_every_half_pattern_widens_exactly():
    """Every binary16 bit pattern the fp16 entry points read is widened to the exact
    binary32 value (compared with torch's CPU conversion, NaNs as NaNs): an eligibility
    trace whose every step terminates returns its inputs unchanged."""
    x = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(HF).reshape(256, 256)
    want = x.float()
    dev = torch.device("cuda")
    term = torch.ones((256, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((256, 256), dtype=torch.float32, device=dev)
    rlca.rlca_eligibility_trace(x.to(dev), term, None, None, decay=0.9, traces=out)
    got = out.cpu()
    nan = torch.isnan(want)
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(got[~nan].view(torch.int32), want[~nan].view(torch.int32))
