"""Structural properties of the oracle's verify (fixed width and per-request
widths) on random small inputs: mixed greedy and sampled requests, random
truncation, non-finite rows and out-of-range proposals anywhere.  Whatever the
inputs, a successful request emits its accepted prefix of proposals and then
exactly one target token; a failed request emits nothing."""
import numpy as np
import pytest
import torch

import synth

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


@settings(max_examples=150, deadline=None)
@given(seed=st.integers(0, 2**32 - 1), V=st.sampled_from([8, 16, 40]), gamma=st.integers(1, 6),
       B=st.integers(1, 6), with_width=st.booleans())
def test_verify_output_structure(oracle, seed, V, gamma, B, with_width):
    rng = np.random.default_rng(seed)
    t = rng.normal(0, 2.0, (B, gamma + 1, V)).astype(np.float32)
    bad = rng.random((B, gamma + 1)) < 0.05
    t[bad, 0] = np.nan
    q = rng.random((B, gamma, V)).astype(np.float32) + 1e-3
    q /= q.sum(-1, keepdims=True)
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    x[rng.random((B, gamma)) < 0.05] = V + 1
    qx = np.take_along_axis(q, np.clip(x, 0, V - 1)[..., None], 2)[..., 0]
    pol = synth.Policy(torch.tensor(rng.uniform(0.5, 1.5, B), dtype=torch.float32),
                       torch.tensor(rng.choice([0, 1, 3, V], B), dtype=torch.int32),
                       torch.tensor(rng.choice([1.0, 0.9, 0.5], B), dtype=torch.float32),
                       torch.tensor(rng.random(B) < 0.3, dtype=torch.int32))
    width = rng.integers(-1, gamma + 2, B).astype(np.int32) if with_width else None
    res = oracle.verify(t, x, q, qx, pol.numpy(), **synth.make_keys(B, seed=seed % 1000).numpy(), width=width)
    for b in range(B):
        out, n, s = res["out_tokens"][b], int(res["num_accepted"][b]), int(res["status"][b])
        w = gamma if width is None else int(width[b])
        if s != 0:
            assert n == -1 and np.all(out == -1), (b, s)
            continue
        assert 0 <= w <= gamma and 0 <= n <= w
        assert np.array_equal(out[:n], x[b, :n])
        assert 0 <= out[n] < V
        assert np.all(out[n + 1:] == -1)
        # a bad width, a proposal checked and out of range, or a NaN in a row
        # the request reads would have failed it
        assert np.all((x[b, :w] >= 0) & (x[b, :w] < V)) and not bad[b, :w + 1].any()
        # the determinate prefix: everything when the request is determinate;
        # otherwise a prefix of the emitted tokens, all of the accepted ones
        # when only the final draw was indeterminate
        dt, dn = int(res["det_tokens"][b]), bool(res["det_nacc"][b])
        if not res["indet"][b]:
            assert dt == gamma + 1 and dn
        elif dn:
            assert dt == n
        else:
            assert 0 <= dt <= n


def test_verify_determinate_prefix_at_a_planted_tie(oracle):
    """Decision 2 planted on its accept threshold (q(x_2) = p_1(x_2) / u_2,
    so u = p/q exactly) after a sure accept of x_1: the oracle marks the
    request indeterminate with x_1 alone still comparable and num_accepted
    undecided."""
    V, gamma, B = 16, 3, 1
    rng = np.random.default_rng(5)
    t = rng.normal(0, 1.0, (B, gamma + 1, V)).astype(np.float32)
    x = np.array([[3, 7, 1]], np.int32)
    q = np.full((B, gamma, V), 1.0 / V, np.float32)
    keys = synth.make_keys(B, seed=4, pos0=10).numpy()
    p1 = torch.softmax(torch.tensor(t[0, 1], dtype=torch.float64), 0).numpy()
    u2 = oracle.uniform(4, 0, 12, 1)
    qx = np.array([[1e-6, np.float32(p1[7] / u2), 0.5]], np.float32)
    pol = synth.uniform_policy(B, temperature=1.0).numpy()
    res = oracle.verify(t, x, q, qx, pol, **keys)
    assert res["indet"][0] and res["det_tokens"][0] == 1 and not res["det_nacc"][0]
    assert res["out_tokens"][0, 0] == 3
    # the same request with decision 2 far from its threshold is determinate
    qx[0, 1] = 1e-6
    res = oracle.verify(t, x, q, qx, pol, **keys)
    if not res["indet"][0]:
        assert res["det_tokens"][0] == gamma + 1 and res["det_nacc"][0]
