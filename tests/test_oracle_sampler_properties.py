"""Structural properties of the oracle's draft samplers (the Markov head and
the RNN head) on random small inputs with mixed policies and non-finite
rows: proposals stop for good at a failure, q(x) is q at the drawn token,
sampled q rows are distributions whose support holds x, greedy requests
report q(x) = 1."""
import numpy as np
import pytest
import torch

import synth

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


def _bf16(a):
    return synth.bf16_bits(torch.tensor(a, dtype=torch.float32).to(torch.bfloat16))


@settings(max_examples=100, deadline=None)
@given(seed=st.integers(0, 2**32 - 1), V=st.sampled_from([8, 24, 64]), gamma=st.integers(1, 5),
       B=st.integers(1, 5), head=st.sampled_from(["markov", "rnn"]))
def test_sampler_output_structure(oracle, seed, V, gamma, B, head):
    rng = np.random.default_rng(seed)
    r = 16
    bb = rng.normal(0, 2.0, (B, gamma, V)).astype(np.float32)
    bad = rng.random((B, gamma)) < 0.05
    bb[bad, 1] = np.inf
    anchor = rng.integers(0, V, B).astype(np.int32)
    anchor[rng.random(B) < 0.1] = -3
    U, W = _bf16(rng.normal(0, 0.5, (V, r))), _bf16(rng.normal(0, 0.5, (V, r)))
    pol = synth.Policy(torch.tensor(rng.uniform(0.5, 1.5, B), dtype=torch.float32),
                       torch.tensor(rng.choice([0, 1, 3, V], B), dtype=torch.int32),
                       torch.tensor(rng.choice([1.0, 0.9, 0.5], B), dtype=torch.float32),
                       torch.tensor(rng.random(B) < 0.3, dtype=torch.int32)).numpy()
    keys = synth.make_keys(B, seed=seed % 1000).numpy()
    if head == "markov":
        res = oracle.markov_sample(bb, anchor, U, W, None, None, None, pol, **keys)
    else:
        Wi, Wh = _bf16(rng.normal(0, 0.3, (3 * r, r))), _bf16(rng.normal(0, 0.3, (3 * r, r)))
        bi, bh = rng.normal(0, 0.1, 3 * r).astype(np.float32), rng.normal(0, 0.1, 3 * r).astype(np.float32)
        res = oracle.rnn_sample(bb, anchor, U, W, Wi, Wh, bi, bh, None, None, None, pol, **keys)
    for b in range(B):
        x, qx, s = res["proposals"][b], res["q_at_x"][b], int(res["status"][b])
        failed = np.nonzero(x < 0)[0]
        first = failed[0] if failed.size else gamma
        assert np.all(x[first:] == -1) and np.all((x[:first] >= 0) & (x[:first] < V))
        assert (s == 0) == (first == gamma)
        if anchor[b] < 0:
            assert s == 5 and first == 0
        for k in range(first):
            if pol["greedy"][b]:
                assert qx[k] == 1.0
            else:
                qk = res["q"][b, k]
                assert abs(float(qk.astype(np.float64).sum()) - 1.0) < 1e-5
                assert qk[x[k]] > 0 and qx[k] == qk[x[k]]
