"""The C-ABI library: it builds, loads, exports every symbol include/*.h declares,
and rejects bad arguments on the host with the documented status codes before any
CUDA call (these tests run without a GPU; the pointers are never dereferenced)."""
import ctypes
import glob
import os
import re

import pytest

import segmented_associative_scan_gb300 as rlca

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

OK, NULL, SHAPE, PARAM, ALIAS, WORKSPACE, LAUNCH, TIMEOUT, MEMORY = 0, -1, -2, -3, -4, -5, -6, -7, -8


@pytest.fixture(scope="module")
def lib():
    rlca.build()
    return rlca.lib()


def declared_functions():
    names = set()
    for header in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(header).read(), flags=re.S)
        names |= set(re.findall(r"\b(rlca_\w+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "rlca_gae" in names and "rlca_retrace" in names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert name in rlca.SIGNATURES, f"{name} has no Python binding"


def test_version_and_status_strings(lib):
    assert lib.rlca_version() >= 100
    for code in (OK, NULL, SHAPE, PARAM, ALIAS, WORKSPACE, LAUNCH, TIMEOUT, MEMORY):
        assert lib.rlca_status_string(code)
    assert b"pinned host memory" in lib.rlca_status_string(MEMORY)
    assert b"unknown" in lib.rlca_status_string(12345)


# Fake, never-dereferenced device addresses, 256 bytes apart per row block.
def fake(i, N=4, T=64):
    return 0x10000000 + i * 0x100000


def gae_args(**kw):
    a = dict(reward=fake(1), value=fake(2), term=fake(3), trunc=None, tv=None, boot=None,
             gamma=0.99, lam=0.95, N=4, T=64, ld=64, adv=fake(4), ret=fake(5), stream=None)
    a.update(kw)
    return (a["reward"], a["value"], a["term"], a["trunc"], a["tv"], a["boot"], a["gamma"],
            a["lam"], a["N"], a["T"], a["ld"], a["adv"], a["ret"], a["stream"])


def test_null_pointers(lib):
    assert lib.rlca_gae(*gae_args(reward=None)) == NULL
    assert lib.rlca_gae(*gae_args(value=None)) == NULL
    assert lib.rlca_gae(*gae_args(term=None)) == NULL
    assert lib.rlca_gae(*gae_args(adv=None)) == NULL
    assert lib.rlca_gae(*gae_args(trunc=fake(6))) == NULL  # truncated without values
    assert lib.rlca_discounted_return(fake(1), fake(2), None, None, None, 0.9, 4, 64, 64,
                                      None, None) == NULL
    assert lib.rlca_retrace(fake(1), fake(2), None, fake(3), fake(4), None, None, None,
                            0.99, 0.95, 4, 64, 64, fake(5), None) == NULL


def test_shapes(lib):
    assert lib.rlca_gae(*gae_args(N=-1)) == SHAPE
    assert lib.rlca_gae(*gae_args(T=-1)) == SHAPE
    assert lib.rlca_gae(*gae_args(ld=63)) == SHAPE
    assert lib.rlca_gae(*gae_args(T=(1 << 30) + 1, ld=(1 << 30) + 1)) == SHAPE
    assert lib.rlca_gae(*gae_args(N=1 << 40, T=1 << 20, ld=1 << 22)) == SHAPE


def test_empty_problems_are_no_ops(lib):
    # N == 0 or T == 0: valid, nothing enqueued, pointers may be NULL.
    assert lib.rlca_gae(*gae_args(N=0, reward=None, value=None, term=None, adv=None)) == OK
    assert lib.rlca_gae(*gae_args(T=0, ld=0, reward=None, adv=None)) == OK
    assert lib.rlca_vtrace(None, None, None, None, None, None, None, 0.99, 1.0, 1.0, 1.0,
                           1.0, 0, 16, 16, None, None, None) == OK


def test_parameters(lib):
    for g in (-0.1, float("nan"), float("inf")):
        assert lib.rlca_gae(*gae_args(gamma=g)) == PARAM
    for lam in (-0.01, 1.01, float("nan")):
        assert lib.rlca_gae(*gae_args(lam=lam)) == PARAM
    assert lib.rlca_td_lambda(fake(1), fake(2), fake(3), None, None, None, 0.9, 2.0, 4, 64,
                              64, fake(4), None) == PARAM
    v = lambda rb, cb, pb: lib.rlca_vtrace(fake(1), fake(2), fake(3), fake(4), None, None,
                                           None, 0.99, 1.0, rb, cb, pb, 4, 64, 64, fake(5),
                                           fake(6), None)
    assert v(0.0, 1.0, 1.0) == PARAM
    assert v(1.0, float("nan"), 1.0) == PARAM
    assert v(1.0, 1.0, -1.0) == PARAM


def test_aliasing(lib):
    N, T = 4, 64
    row_bytes = T * 4
    assert lib.rlca_gae(*gae_args(adv=fake(1))) == ALIAS  # output == reward
    assert lib.rlca_gae(*gae_args(adv=fake(1) + 8)) == ALIAS  # inside reward
    assert lib.rlca_gae(*gae_args(ret=fake(4))) == ALIAS  # two outputs equal
    assert lib.rlca_gae(*gae_args(adv=fake(3) - 16)) == ALIAS  # runs into the flags
    assert lib.rlca_discounted_return(fake(1), fake(2), None, None, fake(3), 0.9, N, T, T,
                                      fake(3) - 8, None) == ALIAS  # overlaps bootstrap


def test_workspace_size_and_validation(lib):
    assert lib.rlca_workspace_bytes(4, 1024) == 0
    assert lib.rlca_workspace_bytes(4, 1025) == 256 + 32 * 4 * 2
    assert lib.rlca_workspace_bytes(2048, 4096) == 256 + 32 * 2048 * 4
    assert lib.rlca_workspace_bytes(-1, 5000) == 0
    N, T = 4, 2048
    need = lib.rlca_workspace_bytes(N, T)
    ws = 0x40000000
    args = lambda w, nb: (fake(1), fake(2), fake(3), None, None, None, 0.99, 0.95, N, T, T,
                          fake(4), fake(5), w, nb, None)
    assert lib.rlca_gae_ex(*args(ws, need - 1)) == WORKSPACE
    assert lib.rlca_gae_ex(*args(ws + 16, need)) == WORKSPACE  # not 256-byte aligned
    assert lib.rlca_gae_ex(*args(fake(1), need)) == ALIAS     # overlaps an input
    assert lib.rlca_gae_ex(*args(fake(4), need)) == ALIAS     # overlaps an output
    assert lib.rlca_testing_lookback_stall(fake(1), fake(2), 4, 1000, fake(3), ws, 10**6, 8,
                                           None) == WORKSPACE  # one tile per row
    assert lib.rlca_workspace_check(None, None) == NULL


def test_td_lambda_multi_validation(lib):
    lam = (ctypes.c_float * 5)(0.0, 0.5, 0.9, 1.0, 0.3)
    outs = (ctypes.c_void_p * 5)(fake(4), fake(5), fake(6), fake(7), fake(8))
    call = lambda n, lams=lam, tg=outs, g=0.99: lib.rlca_td_lambda_multi(
        fake(1), fake(2), fake(3), None, None, None, g, lams, n, 4, 64, 64, tg, None)
    assert call(0) == PARAM and call(5) == PARAM
    assert call(2, lams=None) == NULL and call(2, tg=None) == NULL
    bad = (ctypes.c_float * 2)(0.5, 1.5)
    assert call(2, lams=bad) == PARAM
    assert call(2, g=-1.0) == PARAM
    holes = (ctypes.c_void_p * 3)(fake(4), None, fake(6))
    assert call(3, tg=holes) == NULL
    same = (ctypes.c_void_p * 2)(fake(4), fake(4))
    assert call(2, tg=same) == ALIAS
    into_input = (ctypes.c_void_p * 2)(fake(4), fake(2))
    assert call(2, tg=into_input) == ALIAS


def gae_vtrace_args(**kw):
    a = dict(reward=fake(1), value=fake(2), log_rho=fake(3), term=fake(4), trunc=None,
             tv=None, boot=None, gamma=0.99, lam=0.95, lam_v=1.0, rb=1.0, cb=1.0, pb=1.0,
             N=4, T=64, ld=64, adv=fake(5), ret=fake(6), vs=fake(7), pg=fake(8), stream=None)
    a.update(kw)
    return tuple(a[k] for k in ("reward", "value", "log_rho", "term", "trunc", "tv", "boot",
                                "gamma", "lam", "lam_v", "rb", "cb", "pb", "N", "T", "ld",
                                "adv", "ret", "vs", "pg", "stream"))


def test_gae_vtrace_validation(lib):
    f = lib.rlca_gae_vtrace
    assert f(*gae_vtrace_args(adv=None)) == NULL  # both primary outputs are required
    assert f(*gae_vtrace_args(vs=None)) == NULL
    assert f(*gae_vtrace_args(log_rho=None)) == NULL
    assert f(*gae_vtrace_args(N=0, reward=None, adv=None, vs=None)) == OK  # empty
    assert f(*gae_vtrace_args(lam=1.5)) == PARAM
    assert f(*gae_vtrace_args(lam_v=-0.5)) == PARAM
    assert f(*gae_vtrace_args(cb=0.0)) == PARAM
    assert f(*gae_vtrace_args(vs=fake(5))) == ALIAS  # vs on advantages
    assert f(*gae_vtrace_args(pg=fake(3))) == ALIAS  # pg on log ratios


def test_measure_copy_rejects_bad_arguments(lib):
    """The measurement entry point validates counts, pointers and alignment on the host."""
    arr = lambda *p: (ctypes.c_void_p * max(1, len(p)))(*p)
    ins, fl, outs = arr(fake(1)), arr(fake(2)), arr(fake(3))
    call = lambda i=ins, ni=1, eb=4, f=fl, nf=1, o=outs, no=1, n=1024, c=1: \
        lib.rlca_measure_copy(i, ni, eb, f, nf, o, no, n, c, None)
    assert call(ni=0) == PARAM
    assert call(ni=5) == PARAM
    assert call(nf=3) == PARAM
    assert call(no=0) == PARAM
    assert call(c=3) == PARAM
    assert call(n=-1) == PARAM
    assert call(eb=8) == PARAM
    assert call(i=arr(None)) == NULL
    assert call(i=arr(fake(1) + 16)) == WORKSPACE      # fp32 inputs: 32-byte aligned
    assert call(i=arr(fake(1) + 8), eb=2) == WORKSPACE
    assert call(f=arr(fake(2) + 4)) == WORKSPACE
    assert call(n=0, c=4) == OK
