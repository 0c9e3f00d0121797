"""Host-side checks of the C ABI: the library builds for sm_103a, exports
every entry point include/dspark.h declares, and rejects invalid arguments
before touching device memory (no kernel runs here)."""
import ctypes
import os
import re

import pytest

import verify_dspark_markov_gb300 as ds
from verify_dspark_markov_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dspark.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert len(syms) >= 6
    for s in syms:
        assert hasattr(lib, s), s
    assert set(binding.EXPORTED) == set(syms)


def test_version_and_status_strings(lib):
    assert lib.dspark_version() >= 100
    for code in (0, -1, -2, -3, -4, 1, 2, 3, 4, 5):
        assert ds.status_string(code) and "unknown" not in ds.status_string(code)
    assert "unknown" in ds.status_string(99)


def test_workspace_sizes(lib):
    n1 = ds.workspace_size(ds.OP_VERIFY, 64, 7, 129280)
    n2 = ds.workspace_size(ds.OP_VERIFY, 128, 7, 129280)
    assert 0 < n1 < n2
    assert ds.workspace_size(ds.OP_VERIFY, 64, 0, 129280) == 0      # invalid gamma
    assert ds.workspace_size(ds.OP_VERIFY, 64, 7, 129281) == 0      # V not a multiple of 8
    assert ds.workspace_size(99, 64, 7, 129280) == 0
    # drafting with the Markov bias alternates two fp32 z buffers [B, V]
    assert ds.workspace_size(ds.OP_MARKOV_SAMPLE, 64, 5, 129280, 256) >= 2 * 64 * 129280 * 4
    assert ds.workspace_size(ds.OP_MARKOV_SAMPLE, 64, 5, 129280, 0) < 64 * 129280 * 4


FAKE = ctypes.c_void_p(0x7F0000000000)       # aligned, never dereferenced
FAKE_ODD = ctypes.c_void_p(0x7F0000000004)   # misaligned by 4


def _verify(lib, target=FAKE, dtype=0, B=4, gamma=5, V=1024, ws_bytes=1 << 20, policy=None,
            props=FAKE):
    return lib.dspark_verify(target, dtype, props, FAKE, FAKE, policy, FAKE, FAKE, FAKE, B, gamma, V,
                             FAKE, FAKE, FAKE, FAKE, ws_bytes, None)


def test_verify_rejects_invalid_arguments(lib):
    assert _verify(lib, B=0) == binding.OK                  # empty batch: no-op
    assert _verify(lib, gamma=0) == binding.EINVAL
    assert _verify(lib, gamma=17) == binding.EINVAL
    assert _verify(lib, V=1001) == binding.EINVAL
    assert _verify(lib, V=0) == binding.EINVAL
    assert _verify(lib, B=-1) == binding.EINVAL
    assert _verify(lib, dtype=7) == binding.EINVAL
    assert _verify(lib, target=None) == binding.EINVAL
    assert _verify(lib, props=None) == binding.EINVAL
    assert _verify(lib, target=FAKE_ODD) == binding.EINVAL
    assert _verify(lib, ws_bytes=16, policy=FAKE) == binding.ENOSPC   # sampled path needs workspace


def test_verify_width_rejects_invalid_arguments(lib):
    """dspark_verify_width checks what dspark_verify checks; the widths
    themselves are data (a bad one fails its request, not the call)."""
    def call(B=4, gamma=5, V=1024, target=FAKE, props=FAKE, policy=None, ws_bytes=1 << 20, width=FAKE):
        return lib.dspark_verify_width(target, 0, props, FAKE, FAKE, policy, FAKE, FAKE, FAKE, width, B, gamma,
                                       V, FAKE, FAKE, FAKE, FAKE, ws_bytes, None)
    assert call(B=0) == binding.OK
    assert call(gamma=0) == binding.EINVAL
    assert call(gamma=17) == binding.EINVAL
    assert call(V=1001) == binding.EINVAL
    assert call(target=None) == binding.EINVAL
    assert call(props=None) == binding.EINVAL
    assert call(target=FAKE_ODD) == binding.EINVAL
    assert call(ws_bytes=16, policy=FAKE) == binding.ENOSPC


def test_sts_fit_rejects_invalid_arguments(lib):
    f = lib.dspark_sts_fit
    ws = ds.workspace_size(ds.OP_STS_FIT, 100, 5, 0)
    assert 0 < ws <= 1 << 19
    assert ds.workspace_size(ds.OP_STS_FIT, 100, 0, 0) == 0 and ds.workspace_size(ds.OP_STS_FIT, -1, 5, 0) == 0
    call = lambda N=100, g=5, z=FAKE, a=FAKE, beta=FAKE, st=FAKE, passes=None, mp=0, wsb=ws: f(
        z, a, None, N, g, beta, st, passes, mp, FAKE, wsb, None)
    assert call(g=0) == binding.EINVAL
    assert call(g=17) == binding.EINVAL
    assert call(N=-1) == binding.EINVAL
    assert call(z=None) == binding.EINVAL
    assert call(beta=None) == binding.EINVAL
    assert call(beta=FAKE_ODD) == binding.EINVAL                   # fp64 output, 8-byte aligned
    assert call(z=ctypes.c_void_p(0x7F0000000002)) == binding.EINVAL
    assert call(passes=ctypes.c_void_p(0x7F0000000002)) == binding.EINVAL   # int32 output, 4-byte aligned
    assert call(wsb=8) == binding.ENOSPC
    assert call(mp=-1) == binding.EINVAL                           # pass budget 0 (default) .. 4096
    assert call(mp=4097) == binding.EINVAL


def test_rnn_rejects_invalid_arguments(lib):
    f = lib.dspark_rnn_sample
    ws = ds.workspace_size(ds.OP_RNN_SAMPLE, 4, 5, 1024, 64)
    assert ws >= 2 * 4 * 1024 * 4 and ds.workspace_size(ds.OP_RNN_SAMPLE, 4, 5, 1024, 0) == 0

    def call(B=4, gamma=5, V=1024, r=64, Wi=FAKE, U=FAKE, wsb=ws, policy=None, q=None):
        return f(FAKE, 0, FAKE, U, FAKE, r, Wi, FAKE, FAKE, FAKE, None, 0, None, None, 0, policy, FAKE, FAKE, FAKE,
                 B, gamma, V, FAKE, q, FAKE, None, FAKE, FAKE, wsb, None)
    assert call(B=0) == binding.OK
    assert call(r=0) == binding.EINVAL                      # the RNN head needs a rank
    assert call(r=24) == binding.EINVAL
    assert call(B=300) == binding.EINVAL
    assert call(B=16, V=8) == binding.EINVAL                # the bias gather needs B <= V
    assert call(Wi=None) == binding.EINVAL
    assert call(Wi=FAKE_ODD) == binding.EINVAL
    assert call(policy=FAKE, q=None) == binding.EINVAL
    assert call(wsb=16) == binding.ENOSPC


def _markov(lib, B=4, gamma=5, V=1024, r=0, U=None, W=None, policy=None, q=None, h=None, H=0,
            ws_bytes=1 << 20):
    return lib.dspark_markov_sample(FAKE, 0, FAKE, U, W, r, h, 0, FAKE, FAKE, H, policy, FAKE, FAKE,
                                    FAKE, B, gamma, V, FAKE, q, FAKE, FAKE, FAKE, FAKE, ws_bytes, None)


def test_markov_rejects_invalid_arguments(lib):
    assert _markov(lib, B=0) == binding.OK
    assert _markov(lib, B=257) == binding.EINVAL            # above DSPARK_MAX_BATCH
    assert _markov(lib, r=8, U=FAKE, W=FAKE) == binding.EINVAL      # rank not a multiple of 16
    assert _markov(lib, r=272, U=FAKE, W=FAKE) == binding.EINVAL    # rank above the maximum
    assert _markov(lib, r=16) == binding.EINVAL             # r > 0 without U / W
    assert _markov(lib, r=16, U=FAKE_ODD, W=FAKE) == binding.EINVAL
    assert _markov(lib, policy=FAKE, q=None) == binding.EINVAL      # sampled requests need q
    assert _markov(lib, h=FAKE, H=0) == binding.EINVAL
    assert _markov(lib, ws_bytes=0, policy=FAKE, q=FAKE) == binding.ENOSPC
    assert _markov(lib, ws_bytes=0, r=16, U=FAKE, W=FAKE) == binding.ENOSPC


def test_markov_launch_counts(lib):
    f = lib.dspark_markov_launches
    f.argtypes = [ctypes.c_int] * 7
    f.restype = ctypes.c_int
    assert f(0, 4, 5, 1004, 0, 1, 0) == -1        # V not a multiple of 8
    assert f(0, 257, 5, 1024, 0, 1, 0) == -1      # above DSPARK_MAX_BATCH
    assert f(0, 4, 5, 1024, 8, 1, 0) == -1        # rank not a multiple of 16
    assert f(0, 0, 5, 1024, 0, 1, 1) == 0
    assert f(0, 4, 5, 1024, 0, 0, 0) == 1         # greedy, no bias: one arg-max launch
    assert f(0, 4, 5, 1024, 0, 0, 1) == 2         # ... and the confidence kernel
    assert f(0, 4, 5, 1024, 0, 1, 0) == 5         # sampled, no bias: the policy step per position
    assert f(0, 4, 5, 1024, 16, 1, 1) == 11       # r = 16 (never fused): GEMM + step per position, conf


def test_rnn_launch_counts(lib):
    f = lib.dspark_rnn_launches
    f.argtypes = [ctypes.c_int] * 6
    f.restype = ctypes.c_int
    assert f(0, 4, 5, 1024, 8, 0) == -1           # rank below 16
    assert f(0, 2000, 5, 1024, 16, 0) == -1       # more requests than tokens (and above the maximum)
    assert f(0, 0, 5, 1024, 16, 1) == 0
    assert f(0, 4, 5, 1024, 16, 0) == 20          # r = 16 (never fused): four kernels a step
    assert f(0, 4, 5, 1024, 16, 1) == 21


def test_wait_selftest_rejects_invalid_arguments(lib):
    f = lib.dspark_wait_selftest
    f.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 4
    f.restype = ctypes.c_int
    assert f(0, 0, 1000, FAKE, FAKE, FAKE, None) == binding.EINVAL       # no blocks
    assert f(65, 0, 1000, FAKE, FAKE, FAKE, None) == binding.EINVAL      # more than 64
    assert f(2, -1, 1000, FAKE, FAKE, FAKE, None) == binding.EINVAL      # negative missing arrivals
    assert f(2, 1, 0, FAKE, FAKE, FAKE, None) == binding.EINVAL          # no time limit
    assert f(2, 1, 2_000_001, FAKE, FAKE, FAKE, None) == binding.EINVAL  # above 2 s
    assert f(2, 1, 1000, None, FAKE, FAKE, None) == binding.EINVAL
    assert f(2, 1, 1000, FAKE, FAKE, FAKE_ODD, None) == binding.EINVAL   # workspace not 16-byte aligned


def test_accept_stats_rejects_invalid_arguments(lib):
    f = lib.dspark_accept_stats
    assert f(FAKE, FAKE, 0, FAKE, FAKE, None, 4, 0, 1024, *([FAKE] * 7), FAKE, 1 << 20, None) == binding.EINVAL
    assert f(FAKE, FAKE, 3, FAKE, FAKE, None, 4, 5, 1024, *([FAKE] * 7), FAKE, 1 << 20, None) == binding.EINVAL


def test_accept_stats_grad_rejects_invalid_arguments(lib):
    f = lib.dspark_accept_stats_grad
    args = lambda **kw: dict(dict(d=FAKE, dt=0, N=4, g=5, V=1024, scale=1.0, gd=FAKE), **kw)
    call = lambda a: f(a["d"], FAKE, a["dt"], FAKE, FAKE, None, a["N"], a["g"], a["V"], a["scale"], a["gd"], FAKE,
                       None)
    assert call(args(N=0)) == binding.OK                    # empty batch: no-op
    assert call(args(g=0)) == binding.EINVAL
    assert call(args(V=1001)) == binding.EINVAL
    assert call(args(dt=7)) == binding.EINVAL
    assert call(args(d=None)) == binding.EINVAL
    assert call(args(gd=FAKE_ODD)) == binding.EINVAL        # the gradient rows take 16-byte stores
    assert call(args(scale=float("nan"))) == binding.EINVAL


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises((RuntimeError, OSError)):
        binding._lib = None
        try:
            binding.load(str(tmp_path / "missing.so"))
        finally:
            binding._lib = None
