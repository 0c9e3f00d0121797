"""The Sequential Temperature Scaling root search of the CUDA library
(sts_search.cuh, the code sts_update_kernel runs), compiled for the host and
driven through whole fits: each pass's sums are formed as the pass kernel
forms them (fp32 pair terms at the fp32 beta, fp64 totals) and the searched
beta is compared with the oracle's bisection (status exact, beta within
1e-5; the GPU parity test uses the same bar)."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class StsState(ctypes.Structure):
    _fields_ = [("beta", ctypes.c_double), ("lo", ctypes.c_double), ("hi", ctypes.c_double),
                ("s1", ctypes.c_double), ("s2", ctypes.c_double), ("flags", ctypes.c_uint32),
                ("phase", ctypes.c_int32), ("status", ctypes.c_int32), ("passes", ctypes.c_int32)]


@pytest.fixture(scope="module")
def search(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("shim") / "libsts_search.so")
    cmd = [nvcc, "-std=c++17", "-O2", "-shared", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
           "-gencode", "arch=compute_103a,code=sm_103a",
           f"-I{os.path.join(ROOT, 'include')}", f"-I{os.path.join(ROOT, 'verify_dspark_markov_gb300', 'csrc')}",
           os.path.join(ROOT, "tests", "sts_search_shim.cu"), "-o", out]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.sts_search_step_host.argtypes = [ctypes.POINTER(StsState)]
    lib.sts_search_step_host.restype = ctypes.c_int
    assert lib.sts_state_size() == ctypes.sizeof(StsState)
    return lib


def _fit(lib, z, a, mask=None, passes=64):
    """Whole fits of every position with the library's search; the pass sums
    formed as the device forms them."""
    N, G = z.shape
    m = np.ones((N, G), bool) if mask is None else mask.astype(bool)
    beta, status, used = np.zeros(G), np.zeros(G, np.int32), np.zeros(G, np.int32)
    for k in range(G):
        zk, ak = z[m[:, k], k], a[m[:, k], k]
        st = StsState(beta=0.0, lo=0.0, hi=float("inf"), phase=0)
        flags = 0
        if np.any(~np.isfinite(zk) | ~((ak >= 0) & (ak <= 1))):
            flags |= 4
        if np.any(zk != 0):
            flags |= 1
        if np.any(((zk > 0) & (ak < 1)) | ((zk < 0) & (ak > 0))):
            flags |= 2
        for _ in range(passes):
            b = np.float32(st.beta)
            with np.errstate(over="ignore", invalid="ignore"):
                sg = (np.float32(1) / (np.float32(1) + np.exp(-b * zk))).astype(np.float32)
                t1 = (zk * (sg - ak)).astype(np.float32)
                t2 = (zk * zk * (sg * (np.float32(1) - sg))).astype(np.float32)
            st.s1, st.s2, st.flags = float(t1.astype(np.float64).sum()), float(t2.astype(np.float64).sum()), flags
            if lib.sts_search_step_host(ctypes.byref(st)):
                break
        beta[k], status[k], used[k] = st.beta, st.status, st.passes
    return beta, status, used


def _check(oracle, lib, z, a, mask=None):
    ref = oracle.sts_fit(z, a, mask)
    beta, status, used = _fit(lib, z, a, mask)
    np.testing.assert_array_equal(status, ref["status"])
    fin = np.isfinite(ref["beta"])
    np.testing.assert_allclose(beta[fin], ref["beta"][fin], rtol=1e-5, atol=0)
    assert np.all(np.isnan(beta[~fin]))
    assert used.max() < 64
    return used


def test_search_soft_and_bernoulli_labels(oracle, search):
    rng = np.random.default_rng(21)
    z = rng.normal(0, 2.0, (100_000, 5)).astype(np.float32)
    T = np.array([0.25, 0.5, 1.0, 2.0, 7.0])
    used = _check(oracle, search, z, (1.0 / (1.0 + np.exp(-z.astype(np.float64) / T))).astype(np.float32))
    assert used.max() <= 20  # Newton converges in a handful of passes
    a = (rng.random(z.shape) < 1.0 / (1.0 + np.exp(-z / T))).astype(np.float32)
    _check(oracle, search, z, a, (rng.random(z.shape) < 0.7).astype(np.uint8))


def test_search_degenerate_invalid_and_large_beta(oracle, search):
    rng = np.random.default_rng(22)
    N = 50_000
    z = rng.normal(0, 2.0, (N, 6)).astype(np.float32)
    a = rng.random((N, 6)).astype(np.float32)
    z[:, 0] = 0.0
    a[:, 1] = z[:, 1] > 0
    a[:, 2] = z[:, 2] < 0
    a[:, 4] = 1.0 / (1.0 + np.exp(-z[:, 4]))
    a[:, 5] = np.where(z[:, 5] > 0, 1.0 / (1.0 + np.exp(-z[:, 5])), 0.0)
    mask = np.ones((N, 6), np.uint8)
    mask[:, 3] = 0
    _check(oracle, search, z, a.astype(np.float32), mask)
    z[7, 4] = np.inf
    _check(oracle, search, z, a.astype(np.float32), mask)
    zb = rng.normal(0, 0.01, (N, 2)).astype(np.float32)
    ab = (1.0 / (1.0 + np.exp(-np.clip(zb.astype(np.float64) / np.array([1e-4, 3e-3]), -700, 700)))).astype(np.float32)
    _check(oracle, search, zb, ab)
