"""rlca_gae_noalloc: GAE for callers that cannot allocate device memory (a plugin that a
host framework hands only its input and output buffers, or a loop under a fixed memory
budget where cudaMalloc could fail or stall the device). For long rows and few envs it
runs the look-back path on a static array inside the library; other shapes go to
rlca_gae unchanged.

Checked through the C ABI against the fp64 oracle and against the existing entry point
rlca_gae, on two calls in a row per shape, with shapes that change between calls (the
array keeps the previous call's contents), within the tolerance of the other parity
tests: max|a - b| <= 1e-4 (1 + max|b|). This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr

pytestmark = pytest.mark.gpu

TOL = 1e-4
MAX_TILES = 32768  # RLCA_NOALLOC_MAX_TILES
TILE = 1024        # steps per look-back tile
OK, NULL, SHAPE, PARAM, WORKSPACE = 0, -1, -2, -3, -5


def _ptr(t):
    return None if t is None else t.data_ptr()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _uses_array(N, T):
    """True when the call runs the look-back path on the library's array."""
    return T > TILE and N < 2 * _sms()


def _close(got, want, what):
    got = got.cpu().numpy().astype(np.float64)
    err = np.max(np.abs(got - want))
    assert err <= TOL * (1.0 + np.max(np.abs(want))), f"{what}: max|err| {err:.3e}"


class _Case:
    """One seeded GAE batch on the device, its oracle result and rlca_gae's."""

    def __init__(self, N, T, dev):
        rlca.build()
        self.lib = rlca.lib()
        ro = sr.gae_trunc(N=N, T=T, seed=N + T)
        self.N, self.T = N, T
        self.g, self.lam = ro.params["gamma"], ro.params["lam"]
        d = lambda a: torch.from_numpy(a).to(dev)
        self.inputs = [d(ro.reward), d(ro.value), d(ro.terminated), d(ro.truncated),
                       d(ro.trunc_value), d(ro.bootstrap)]
        self.want = oracle.gae(ro.reward, ro.value, ro.terminated, ro.truncated,
                               ro.trunc_value, ro.bootstrap, gamma=self.g, lam=self.lam)
        self.stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        self.dev = dev
        self.ref = self.run(self.lib.rlca_gae)

    def run(self, fn):
        adv = torch.full((self.N, self.T), float("nan"), device=self.dev)
        ret = torch.full((self.N, self.T), float("nan"), device=self.dev)
        st = fn(*map(_ptr, self.inputs), self.g, self.lam, self.N, self.T, self.T,
                adv.data_ptr(), ret.data_ptr(), self.stream)
        assert st == OK, f"status {st}"
        torch.cuda.synchronize()
        return adv, ret

    def check_noalloc(self, what):
        adv, ret = self.run(self.lib.rlca_gae_noalloc)
        for got, want, ref, name in zip((adv, ret), self.want, self.ref, ("adv", "ret")):
            _close(got, want, f"{what} {name} vs oracle")
            _close(got, ref.cpu().numpy().astype(np.float64), f"{what} {name} vs rlca_gae")


def test_noalloc_reuses_its_array_across_shapes(cuda_device):
    """Two calls in a row per shape, the shape changing between pairs: every call here
    runs look-back on the library's array, which keeps the previous call's state."""
    shapes = [(64, 5000), (200, 3000), (64, 5000), (5, 70000)]
    assert all(_uses_array(N, T) for N, T in shapes)
    cases = {s: _Case(*s, cuda_device) for s in set(shapes)}
    for k, s in enumerate(shapes):
        for call in range(2):
            cases[s].check_noalloc(f"shape {s}, pair {k}, call {call}")


def test_noalloc_at_its_exact_tile_limit(cuda_device):
    """N * ceil(T / 1024) == RLCA_NOALLOC_MAX_TILES fills the array exactly."""
    N, T = 256, (MAX_TILES // 256) * TILE
    assert _uses_array(N, T) and N * (T // TILE) == MAX_TILES
    case = _Case(N, T, cuda_device)
    case.check_noalloc("limit, call 0")
    case.check_noalloc("limit, call 1")


@pytest.mark.parametrize("N,T", [(16384, 4096), (300, 1000)])
def test_noalloc_shapes_without_look_back_match_gae(cuda_device, N, T):
    """Enough rows to fill the GPU (any number of tiles), or rows of one tile: the call
    is rlca_gae's own, with no workspace, whatever the array's size."""
    assert not _uses_array(N, T)
    case = _Case(N, T, cuda_device)
    case.check_noalloc(f"[{N}, {T}], call 0")
    case.check_noalloc(f"[{N}, {T}], call 1")


def test_noalloc_rejects_look_back_beyond_its_array(cuda_device):
    rlca.build()
    lib = rlca.lib()
    fake = 1 << 40  # never dereferenced: every rejection comes before a launch
    ptrs = lambda: (fake, fake + (1 << 36), fake + (2 << 36), None, None, None)
    out = fake + (3 << 36)
    # The most rows that still take look-back, one tile per row more than fits.
    N = 2 * _sms() - 1
    T = (MAX_TILES // N + 1) * TILE
    assert N * (T // TILE) > MAX_TILES
    assert lib.rlca_gae_noalloc(*ptrs(), 0.99, 0.95, N, T, T, out, None, None) == WORKSPACE
    # Errors of rlca_gae's checks come first, in its order.
    assert lib.rlca_gae_noalloc(*ptrs(), 0.99, 0.95, -1, T, T, out, None, None) == SHAPE
    assert lib.rlca_gae_noalloc(*ptrs(), 0.99, 0.95, N, T, T - 1, out, None, None) == SHAPE
    assert lib.rlca_gae_noalloc(*ptrs(), float("nan"), 0.95, N, T, T, out, None,
                                None) == PARAM
    assert lib.rlca_gae_noalloc(None, *ptrs()[1:], 0.99, 0.95, N, T, T, out, None,
                                None) == NULL
