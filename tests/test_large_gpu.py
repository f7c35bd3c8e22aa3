"""Sizes past 2^31 elements: every offset must be 64-bit. Inputs are drawn on the device
from a seeded generator (N(0,1) data, Bernoulli flags); sampled rows, including the
last rows with the largest offsets, are compared with the fp64 oracle run on those
rows alone. About 50 GB of device memory at most."""
import numpy as np
import pytest
import torch

import oracle
import segmented_associative_scan_gb300 as rlca
from parity_helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()
    yield
    torch.cuda.empty_cache()


def _draw(N, T, seed, trunc=True):
    g = torch.Generator(device="cuda").manual_seed(seed)
    d = dict(reward=torch.randn((N, T), generator=g, device="cuda"),
             value=torch.randn((N, T), generator=g, device="cuda"),
             bootstrap=torch.randn((N,), generator=g, device="cuda"))
    d["terminated"] = (torch.rand((N, T), generator=g, device="cuda") < 2e-3).to(torch.uint8)
    if trunc:
        u = torch.rand((N, T), generator=g, device="cuda")
        d["truncated"] = ((u < 1e-3) & (d["terminated"] == 0)).to(torch.uint8)
        d["trunc_value"] = torch.randn((N, T), generator=g, device="cuda")
    return d


def _rows(d, rows):
    return {k: v[rows].cpu().numpy() for k, v in d.items()}


def test_gae_past_2_31_elements():
    N, T = 2049, 1 << 20  # 2.15e9 steps
    assert N * T > 2 ** 31
    d = _draw(N, T, seed=1)
    adv, ret = rlca.rlca_gae(d["reward"], d["value"], d["terminated"], d["truncated"],
                             d["trunc_value"], d["bootstrap"], gamma=0.99, lam=0.95)
    torch.cuda.synchronize()
    rows = [0, 1, 1024, 2047, 2048]
    h = _rows(d, rows)
    ref_adv, ref_ret = oracle.gae(h["reward"], h["value"], h["terminated"], h["truncated"],
                                  h["trunc_value"], h["bootstrap"], gamma=0.99, lam=0.95)
    assert_parity({"adv": adv[rows].cpu().numpy().astype(np.float64),
                   "ret": ret[rows].cpu().numpy().astype(np.float64)},
                  {"adv": ref_adv, "ret": ref_ret}, "gae 2049 x 2^20")


def test_return_past_2_31_elements_with_padded_rows():
    N, T, ld = 2050, (1 << 20) + 3, (1 << 20) + 8  # ragged rows, padded stride
    assert N * ld > 2 ** 31
    d = _draw(N, ld, seed=2, trunc=False)
    r, term = d["reward"][:, :T], d["terminated"][:, :T]
    out = torch.full((N, ld), -7.0, device="cuda")
    rlca.rlca_discounted_return(r, term, bootstrap=d["bootstrap"], gamma=0.999,
                                returns=out[:, :T])
    torch.cuda.synchronize()
    rows = [0, 1025, 2049]
    ref = oracle.discounted_return(r[rows].cpu().numpy(), term[rows].cpu().numpy(),
                                   bootstrap=d["bootstrap"][rows].cpu().numpy(), gamma=0.999)
    assert_parity({"g": out[rows, :T].cpu().numpy().astype(np.float64)}, {"g": ref},
                  "return 2050 x (2^20+3)")
    assert bool((out[:, T:] == -7.0).all())  # padding columns untouched


def test_lookback_with_rows_of_2_26_steps():
    N, T = 3, 1 << 26  # 2^16 tiles per row, one CTA per tile
    d = _draw(N, T, seed=3)
    ws = rlca.make_workspace(N, T)
    adv, _ = rlca.rlca_gae(d["reward"], d["value"], d["terminated"], d["truncated"],
                           d["trunc_value"], d["bootstrap"], gamma=0.99, lam=0.95,
                           workspace=ws)
    assert rlca.workspace_check(ws) == 0
    h = _rows(d, [0, 1, 2])
    ref, _ = oracle.gae(h["reward"], h["value"], h["terminated"], h["truncated"],
                        h["trunc_value"], h["bootstrap"], gamma=0.99, lam=0.95)
    assert_parity({"adv": adv.cpu().numpy().astype(np.float64)}, {"adv": ref},
                  "gae look-back 3 x 2^26")
