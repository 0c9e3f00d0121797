"""The allocation-free greedy verify (dspark_verify_greedy_noalloc).

It serves callers that cannot allocate device memory for scratch (a plugin
whose host runtime owns all device memory, or a path that must not call
cudaMalloc).  The greedy kernel keeps its state on chip, so neither this entry
point nor dspark_verify with policy NULL needs a workspace.  This file is
named to be collected last.  It builds and loads the library itself, so it
also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from verify_dspark_markov_gb300 import binding, build
    build.build()
    L = binding.load()
    P, i32 = ctypes.c_void_p, ctypes.c_int
    L.dspark_verify_greedy_noalloc.argtypes = [P, i32, P, i32, i32, i32, P, P, P, P]
    L.dspark_verify_greedy_noalloc.restype = i32
    return L


def _noalloc(L, target, proposals):
    B, rows, V = target.shape
    out = torch.full((B, rows), -9, dtype=torch.int32, device=target.device)
    nacc = torch.full((B,), -9, dtype=torch.int32, device=target.device)
    st = torch.full((B,), -9, dtype=torch.int32, device=target.device)
    P = ctypes.c_void_p
    code = L.dspark_verify_greedy_noalloc(
        P(target.data_ptr()), 0 if target.dtype == torch.bfloat16 else 1, P(proposals.data_ptr()),
        B, rows - 1, V, P(out.data_ptr()), P(nacc.data_ptr()), P(st.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))
    assert code == 0, code
    return out, nacc, st


def test_noalloc_matches_verify_twice_in_a_row(lib):
    import verify_dspark_markov_gb300 as ds
    w = synth.full_decode_tile(device="cuda")
    x = w.backbone.float().argmax(dim=2).to(torch.int32)
    ref = ds.verify(w.target, x)
    for _ in range(2):
        got = _noalloc(lib, w.target, x)
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    # a call of another shape right after, on the same stream: it must match
    # dspark_verify too
    w2 = synth.full_decode_tile(V=40_008, B=9, gamma=3, device="cuda", seed=77)
    x2 = w2.backbone.float().argmax(dim=2).to(torch.int32)
    x2[0, 1] = 5
    ref2 = ds.verify(w2.target, x2)
    got2 = _noalloc(lib, w2.target, x2)
    torch.cuda.synchronize()
    for a, b in zip(ref2, got2):
        assert torch.equal(a, b)


def test_noalloc_large_batch_and_no_workspace(lib):
    """A batch above DSPARK_MAX_BATCH (the greedy verify has no batch limit),
    and dspark_verify itself called with a NULL workspace of 0 bytes: both
    match the binding's dspark_verify."""
    import verify_dspark_markov_gb300 as ds
    w = synth.full_decode_tile(V=4096, B=300, gamma=3, device="cuda", seed=5)
    x = w.backbone.float().argmax(dim=2).to(torch.int32)
    x[::7, 1] = 3
    ref = ds.verify(w.target, x)
    got = _noalloc(lib, w.target, x)
    B, rows, V = w.target.shape
    out = torch.full((B, rows), -9, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    st = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    code = lib.dspark_verify(P(w.target.data_ptr()), 0, P(x.data_ptr()), None, None, None, None, None, None,
                             B, rows - 1, V, P(out.data_ptr()), P(nacc.data_ptr()), P(st.data_ptr()), None, 0,
                             P(torch.cuda.current_stream().cuda_stream))
    assert code == 0, code
    torch.cuda.synchronize()
    for a, b, c in zip(ref, got, (out, nacc, st)):
        assert torch.equal(a, b)
        assert torch.equal(a, c)
    assert int((ref[1] < rows - 1).sum()) > 0      # some requests stop early


def test_noalloc_overlapping_streams(lib):
    """Two calls with different batches enqueued on two streams with no
    synchronisation between them (they may run at the same time on the GPU):
    each matches dspark_verify on its own batch."""
    import verify_dspark_markov_gb300 as ds
    cases = []
    for seed, (V, B, gamma) in ((11, (40_008, 33, 5)), (12, (8192, 70, 7))):
        w = synth.full_decode_tile(V=V, B=B, gamma=gamma, device="cuda", seed=seed)
        x = w.backbone.float().argmax(dim=2).to(torch.int32)
        x[::5, 0] = 1
        cases.append((w.target, x, ds.verify(w.target, x)))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = []
    for (t, x, _), s in zip(cases, streams):
        with torch.cuda.stream(s):
            got.append(_noalloc(lib, t, x))
    torch.cuda.synchronize()
    for (_, _, ref), g in zip(cases, got):
        for a, b in zip(ref, g):
            assert torch.equal(a, b)
