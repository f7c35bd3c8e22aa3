"""GPU parity of the pipelined warp-owned rows: a warp per row that asks for the raw words
of its next chunks before it scans the current one. The dispatch takes it for fp32 GAE
with truncation (or rows of at most 512 steps) and for every estimator with bf16 inputs,
on rows longer than one warp chunk (256 steps; bf16 estimators other than GAE: two) up
to 1024 steps, in device memory with 16-byte aligned rows. A row whose length is not a
multiple of the warp chunk starts with a ragged chunk scanned on its own; the rest of the
row, or a whole full row, runs through the pipeline. Covers 2-4 chunks per row, ragged
first chunks of 1-255 steps, padded and offset layouts, 64-bit and 32-bit flag loads,
and the fp64 oracle as reference with the same tolerance as the other parity tests."""
import pytest
import torch

import segmented_associative_scan_gb300 as rlca
import synthetic_rollouts as sr
from parity_helpers import ESTIMATORS, assert_parity, bf16_rounded, run_gpu, run_oracle

pytestmark = pytest.mark.gpu
BF = torch.bfloat16

T_PIPE = [257, 263, 511, 512, 513, 640, 768, 1000, 1016, 1023, 1024]


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()


@pytest.mark.parametrize("trunc", [True, False])
@pytest.mark.parametrize("N", [1, 6, 37])
@pytest.mark.parametrize("T", T_PIPE)
def test_gae_fp32(T, N, trunc):
    ro = sr.generic(N, T, seed=1000 + 7 * N + T, p_term=0.01, p_trunc=0.01 if trunc else 0.0)
    if not trunc:
        ro.truncated = None
    assert_parity(run_gpu("gae", ro, {}), run_oracle("gae", ro, {}),
                  f"gae N={N} T={T} trunc={trunc}")


@pytest.mark.parametrize("ld_extra,offset", [(4, 0), (8, 0), (0, 4), (12, 8), (3, 0)])
@pytest.mark.parametrize("T", [264, 520, 1000, 1024])
def test_gae_fp32_layouts(T, ld_extra, offset):
    """128-bit rows (ld % 8 == 4 or a 16-byte offset), 32-byte rows, and (ld odd) the
    scalar warp-owned rows instead of the pipeline."""
    ro = sr.generic(9, T, seed=2000 + T + ld_extra + offset, p_term=0.01, p_trunc=0.01)
    assert_parity(run_gpu("gae", ro, {}, ld=T + ld_extra, offset=offset),
                  run_oracle("gae", ro, {}), f"gae T={T} ld+{ld_extra} off={offset}")


@pytest.mark.parametrize("trunc", [True, False])
@pytest.mark.parametrize("T", [257, 300, 520, 777, 1016, 1024])
def test_bf16_estimators(T, trunc):
    ro = bf16_rounded(sr.generic(21, T, seed=3000 + T, p_term=0.01,
                                 p_trunc=0.01 if trunc else 0.0))
    if not trunc:
        ro.truncated = None
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, in_dtype=BF), run_oracle(est, ro, {}),
                      f"{est} bf16 T={T} trunc={trunc}")


@pytest.mark.parametrize("T", [520, 1024])
def test_bf16_outputs_off_32_bytes(T):
    """Outputs 16 bytes past a 32-byte boundary: rows fit 128-bit access but not the
    32-byte level, so flags are read 4 bytes at a time instead of 8."""
    ro = bf16_rounded(sr.generic(13, T, seed=4000 + T, p_term=0.01, p_trunc=0.01))
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, in_dtype=BF, out_offset=4),
                      run_oracle(est, ro, {}), f"{est} bf16 T={T} outputs +16 B")


@pytest.mark.parametrize("params", [dict(gamma=1.0, lam=1.0), dict(lam=0.0),
                                    dict(gamma=0.0)])
def test_parameters(params):
    ro = sr.generic(7, 1000, seed=5000, p_term=0.01, p_trunc=0.01)
    assert_parity(run_gpu("gae", ro, params), run_oracle("gae", ro, params), f"gae {params}")
    rb = bf16_rounded(ro)
    for est in ESTIMATORS:
        q = {k: v for k, v in params.items() if est != "return" or k == "gamma"}
        assert_parity(run_gpu(est, rb, q, in_dtype=BF), run_oracle(est, rb, q),
                      f"{est} bf16 {q}")


@pytest.mark.parametrize("ld_extra,offset", [(0, 0), (8, 0), (4, 0), (0, 4)])
@pytest.mark.parametrize("N", [9001, 12288])
def test_rows_walked_by_one_wave(N, ld_extra, offset):
    """Rows of exactly 256 steps, more of them than one wave of warps holds: one wave of
    warps walks the rows, each loading its next row while it scans the current one. Row
    counts that do not divide the grid, and padded or offset layouts."""
    ro = sr.generic(N, 256, seed=6000 + N + ld_extra, p_term=0.01, p_trunc=0.01)
    for est in ESTIMATORS:
        assert_parity(run_gpu(est, ro, {}, ld=256 + ld_extra, offset=offset),
                      run_oracle(est, ro, {}), f"{est} N={N} ld+{ld_extra} off={offset}")


@pytest.mark.parametrize("N,T", [(20000, 128), (40000, 64), (20002, 128)])
def test_packed_rows_walked_by_one_wave(N, T):
    """Rows of 128 or 64 steps packed two or four to a warp chunk (contiguous, ld == T),
    more such jobs than one wave holds: the walked rows. An odd number of jobs per warp
    and, for [20002, 128], jobs that do not divide the grid."""
    ro = sr.generic(N, T, seed=7000 + N + T, p_term=0.02, p_trunc=0.01)
    for est in ("return", "td_lambda", "gae"):
        assert_parity(run_gpu(est, ro, {}), run_oracle(est, ro, {}), f"{est} N={N} T={T}")


@pytest.mark.parametrize("fmt", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("N,T", [(40, 128), (9001, 256), (20000, 128), (37, 1024), (9, 2100)])
def test_bootstrap_read_early_or_late(N, T, fmt):
    """The per-env bootstrap is read beside a chunk's data on some paths and only once the
    flags are in on others (the row loops, some pipelined rows). Every layout (warp-owned
    rows, walked rows, pipelined or CTA rows, the row loop) in every input format: without
    a bootstrap, and with one while the last step is truncated (its truncation value wins)
    or terminated (no successor value)."""
    from parity_helpers import fp16_rounded
    dtype = {"fp32": torch.float32, "bf16": BF, "fp16": torch.float16}[fmt]
    rnd = {"fp32": lambda r: r, "bf16": bf16_rounded, "fp16": fp16_rounded}[fmt]
    for case in ("no bootstrap", "truncated last step", "terminated last step"):
        ro = rnd(sr.generic(N, T, seed=8000 + N + T, p_term=0.01, p_trunc=0.01))
        if case == "no bootstrap":
            ro.bootstrap = None
        elif case == "truncated last step":
            ro.truncated[::2, -1] = 1
        else:
            ro.terminated[1::2, -1] = 1
        for est in ESTIMATORS:
            assert_parity(run_gpu(est, ro, {}, in_dtype=dtype), run_oracle(est, ro, {}),
                          f"{est} {fmt} N={N} T={T} {case}")


@pytest.mark.parametrize("N", [37, 4096, 5000])
@pytest.mark.parametrize("T", [513, 600, 768, 900, 960, 961, 1024])
def test_fp32_return_rows_by_length(N, T):
    """The fp32 discounted return on rows of 513-960 steps takes the pipelined warp rows
    (two chunks in flight, 7 CTAs per SM) while one wave holds them, the CTA row
    otherwise (longer rows, N = 5000): both against the oracle."""
    ro = sr.generic(N, T, seed=9000 + N + T, p_term=0.01, p_trunc=0.01)
    assert_parity(run_gpu("return", ro, {}), run_oracle("return", ro, {}),
                  f"return N={N} T={T}")
