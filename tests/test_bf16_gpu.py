"""GPU parity of the bf16-input entry points: every per-step data input is rounded to
bf16 first, the kernels widen each value to fp32 exactly and compute in fp32, and the
result is compared with the fp64 oracle on the same widened values (same tolerance as
the fp32 paths). Covers warp-owned rows, CTA tiles, the row loop, the forward scans,
strided and unaligned layouts."""
import numpy as np
import pytest
import torch

import oracle
import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr
from parity_helpers import (ESTIMATORS, SENTINEL, Placed, assert_parity, bf16_rounded,
                            run_gpu, run_oracle)

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()


@pytest.mark.parametrize("T", [1, 7, 128, 256, 300, 1024, 1100, 4096])
def test_bf16_reverse_estimators(T):
    ro = bf16_rounded(sr.generic(9, T, seed=T, p_term=0.02, p_trunc=0.01))
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, in_dtype=BF), run_oracle(est, ro, {}),
                      f"{est} bf16 T={T}")


@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (8, 0), (4, 0), (0, 2), (3, 1)])
def test_bf16_layouts(ld_extra, offset):
    """ld % 8 == 0 with aligned bases takes 128-bit loads; the rest the scalar path."""
    ro = bf16_rounded(sr.generic(4, 1000, seed=3))
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, ld=1000 + ld_extra, offset=offset, in_dtype=BF),
                      run_oracle(est, ro, {}), f"{est} bf16 ld+{ld_extra} off={offset}")


@pytest.mark.parametrize("trunc", [True, False])
@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (16, 0), (16, 8)])
@pytest.mark.parametrize("T", [272, 512, 768, 1024])
def test_bf16_gae_rows(T, ld_extra, offset, trunc):
    """bf16 GAE on rows of 257-1024 steps (pipelined warp-owned rows), with and without
    truncation, on padded and offset layouts."""
    ro = bf16_rounded(sr.generic(40, T, seed=T + ld_extra + offset, p_term=0.01,
                                 p_trunc=0.005 if trunc else 0.0))
    if not trunc:
        ro.truncated = None
    assert_parity(run_gpu("gae", ro, {}, ld=T + ld_extra, offset=offset,
                          in_dtype=torch.bfloat16),
                  run_oracle("gae", ro, {}), f"gae bf16 T={T} ld+{ld_extra} off={offset}")


def test_bf16_workloads():
    for est, ro, p in (("gae", sr.gae_trunc(), dict(gamma=0.995, lam=0.95)),
                       ("vtrace", sr.vtrace(), dict(gamma=0.99, lam=1.0)),
                       ("retrace", sr.retrace(N=512), dict(gamma=0.99, lam=0.95))):
        ro = bf16_rounded(ro)
        assert_parity(run_gpu(est, ro, p, in_dtype=BF), run_oracle(est, ro, p), f"{est} bf16")


@pytest.mark.parametrize("T", [5, 200, 1024, 3000])
def test_bf16_forward_scans(T):
    ro = bf16_rounded(sr.generic(6, T, seed=T + 1, p_term=0.02, p_trunc=0.01))
    dev = "cuda:0"
    x = torch.from_numpy(ro.value).to(dev).to(BF)
    d = torch.from_numpy(ro.terminated).to(dev)
    tr = torch.from_numpy(ro.truncated).to(dev)
    init = torch.from_numpy(ro.bootstrap).to(dev)
    got = rlca.rlca_eligibility_trace(x, d, tr, init, decay=0.9)
    ref = oracle.eligibility_trace(ro.value, ro.terminated, ro.truncated, ro.bootstrap, decay=0.9)
    assert_parity({"o": got.cpu().numpy().astype(np.float64)}, {"o": ref}, f"trace T={T}")
    got = rlca.rlca_episodic_prefix_sum(x, d, tr, init)
    ref = oracle.episodic_prefix_sum(ro.value, ro.terminated, ro.truncated, ro.bootstrap)
    assert_parity({"o": got.cpu().numpy().astype(np.float64)}, {"o": ref}, f"sum T={T}")


def test_bf16_rejects_mixed_dtypes_and_workspace():
    dev = "cuda:0"
    r = torch.zeros((4, 2048), device=dev, dtype=BF)
    v = torch.zeros((4, 2048), device=dev, dtype=torch.float32)
    d = torch.zeros((4, 2048), device=dev, dtype=torch.uint8)
    with pytest.raises(TypeError):
        rlca.rlca_gae(r, v, d)
    with pytest.raises(ValueError):
        rlca.rlca_gae(r, r, d, workspace=torch.zeros(4096, dtype=torch.uint8, device=dev))
