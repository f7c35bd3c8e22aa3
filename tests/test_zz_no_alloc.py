"""rlca_gae_noalloc: GAE for callers that cannot allocate device memory (a plugin that a
host framework hands only its input and output buffers, or a loop under a fixed memory
budget where cudaMalloc could fail or stall the device). For long rows it runs the
look-back path on a static workspace inside the library.

Checked through the C ABI against the existing entry point rlca_gae, on two calls in a
row (the second reuses the static workspace the first one left behind), within the
tolerance of the other parity tests: max|a - b| <= 1e-4 (1 + max|b|). This file is
collected last."""
import ctypes

import numpy as np
import pytest
import torch

import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr

pytestmark = pytest.mark.gpu

TOL = 1e-4
MAX_TILES = 32768  # RLCA_NOALLOC_MAX_TILES


def _ptr(t):
    return None if t is None else t.data_ptr()


def _gae_args(ro, dev):
    d = lambda a: None if a is None else torch.from_numpy(a).to(dev)
    return [d(ro.reward), d(ro.value), d(ro.terminated), d(ro.truncated),
            d(ro.trunc_value), d(ro.bootstrap)]


@pytest.mark.parametrize("N,T", [(64, 5000), (2048, 4096), (300, 1000)])
def test_noalloc_matches_gae_on_two_calls(cuda_device, N, T):
    rlca.build()
    lib = rlca.lib()
    ro = sr.gae_trunc(N=N, T=T, seed=N + T)
    g, lam = ro.params["gamma"], ro.params["lam"]
    inputs = _gae_args(ro, cuda_device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ref_adv = torch.empty((N, T), device=cuda_device)
    ref_ret = torch.empty_like(ref_adv)
    assert lib.rlca_gae(*map(_ptr, inputs), g, lam, N, T, T, ref_adv.data_ptr(),
                        ref_ret.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    ref = [ref_adv.cpu().numpy().astype(np.float64), ref_ret.cpu().numpy().astype(np.float64)]

    for call in range(2):
        adv = torch.full((N, T), float("nan"), device=cuda_device)
        ret = torch.full((N, T), float("nan"), device=cuda_device)
        assert lib.rlca_gae_noalloc(*map(_ptr, inputs), g, lam, N, T, T, adv.data_ptr(),
                                    ret.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        for got, want in zip((adv, ret), ref):
            got = got.cpu().numpy().astype(np.float64)
            err = np.max(np.abs(got - want))
            assert err <= TOL * (1.0 + np.max(np.abs(want))), f"call {call}: {err:.3e}"


def test_noalloc_rejects_sizes_beyond_its_static_workspace(cuda_device):
    rlca.build()
    lib = rlca.lib()
    N, T = MAX_TILES // 4 + 1, 4096  # one tile more than the static workspace holds
    fake = 1 << 40  # never dereferenced: the size check comes first
    assert lib.rlca_gae_noalloc(fake, fake + (1 << 36), fake + (2 << 36), None, None, None,
                                0.99, 0.95, N, T, T, fake + (3 << 36), None, None) == -5
