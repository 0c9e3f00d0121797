"""Pins of the oracle's verify over a per-request width (the number of
proposals a request checks, 0..gamma; the pages choose it from measured draft
and verify costs, so it is an input here): the emitted tokens keep the law of
target-only sampling at every width, the bonus comes from the row after the
last checked proposal, and rows or proposals past the width are never read."""
import numpy as np
import pytest
import torch

import synth


def _softmax64(z):
    return torch.softmax(torch.tensor(z, dtype=torch.float64), dim=0).numpy()


def _regime(regime, rng, gamma, V):
    t_logits = rng.normal(0, 1.5, (gamma + 1, V))
    if regime == "agreeing":
        d_logits = t_logits[:gamma] + rng.normal(0, 0.3, (gamma, V))
    elif regime == "disagreeing":
        d_logits = rng.normal(0, 1.5, (gamma, V))
    else:  # nearly disjoint
        t_logits[:, 4:] = -np.inf
        d_logits = np.full((gamma, V), 0.0)
        d_logits[:, :4] = -6.0
    return t_logits, d_logits


def _run(oracle, t_logits, d_logits, width, B, seed):
    gamma, V = d_logits.shape
    rng = np.random.default_rng(seed + 1)
    t = np.tile(t_logits.astype(np.float32), (B, 1, 1))
    q_rows = np.stack([_softmax64(d_logits[k]) for k in range(gamma)])
    q = np.tile(q_rows.astype(np.float32), (B, 1, 1))
    x = np.stack([rng.choice(V, size=B, p=q_rows[k] / q_rows[k].sum()) for k in range(gamma)], 1).astype(np.int32)
    qx = np.take_along_axis(q, x[..., None], 2)[..., 0]
    pol = synth.uniform_policy(B).numpy()
    return oracle.verify(t, x, q, qx, pol, **synth.make_keys(B, seed=seed).numpy(),
                         width=np.full(B, width, np.int32))


def _law(tokens, p):
    from scipy import stats
    sup = p > 0
    assert np.all(sup[tokens])
    if sup.sum() == 1:
        assert np.all(tokens == np.argmax(p))
        return
    c = np.bincount(tokens, minlength=len(p))[sup]
    assert stats.chisquare(c, p[sup] * c.sum()).pvalue > 1e-3


@pytest.mark.parametrize("regime", ["agreeing", "disagreeing", "nearly_disjoint"])
def test_width_preserves_target_law(oracle, regime):
    """Width 2 of gamma = 3 (chi-square, alpha = 1e-3): the first emitted token
    ~ p_0; with both proposals accepted the extra token ~ p_2, the row after
    the last checked proposal (not row gamma); never more than 2 accepted."""
    V, gamma, B = 8, 3, 200_000
    rng = np.random.default_rng({"agreeing": 21, "disagreeing": 22, "nearly_disjoint": 23}[regime])
    t_logits, d_logits = _regime(regime, rng, gamma, V)
    res = _run(oracle, t_logits, d_logits, 2, B, seed=31)
    assert np.all(res["status"] == 0) and np.all(res["num_accepted"] <= 2)
    assert np.all(res["out_tokens"][:, 3] == -1)
    _law(res["out_tokens"][:, 0], _softmax64(t_logits[0]))
    sel = res["num_accepted"] == 2
    if sel.sum() > 2000:
        _law(res["out_tokens"][sel, 2], _softmax64(t_logits[2]))


def test_width_zero_is_target_only_sampling(oracle):
    """Width 0: no proposal is checked, one token is drawn from row 0."""
    V, gamma, B = 8, 3, 200_000
    rng = np.random.default_rng(24)
    t_logits, d_logits = _regime("disagreeing", rng, gamma, V)
    res = _run(oracle, t_logits, d_logits, 0, B, seed=32)
    assert np.all(res["num_accepted"] == 0) and np.all(res["out_tokens"][:, 1:] == -1)
    _law(res["out_tokens"][:, 0], _softmax64(t_logits[0]))


def test_width_gamma_is_the_fixed_width_verify(oracle):
    """Every request at width gamma reproduces the fixed-width verify."""
    w = synth.decode_verify_tile(V=512, B=24, r=0, H=0)
    d = oracle.markov_sample(synth.host(w.backbone), w.anchor.cpu().numpy(), None, None, None, None, None,
                             w.policy.numpy(), **w.keys.numpy())
    args = (synth.host(w.target), d["proposals"], d["q"], d["q_at_x"], w.policy.numpy())
    a = oracle.verify(*args, **w.keys.numpy())
    b = oracle.verify(*args, **w.keys.numpy(), width=np.full(w.B, w.gamma, np.int32))
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_width_greedy_prefix(oracle):
    """Greedy: the matching prefix stops at the width, then the argmax of the
    next row; width 0 emits the argmax of row 0."""
    V, gamma, B = 16, 5, 3
    rng = np.random.default_rng(25)
    t = rng.normal(0, 1, (B, gamma + 1, V)).astype(np.float32)
    am = t.argmax(-1)
    x = am[:, :gamma].astype(np.int32)  # every proposal matches
    pol = synth.uniform_policy(B, greedy=True).numpy()
    res = oracle.verify(t, x, None, None, pol, **synth.make_keys(B).numpy(), width=np.array([2, 0, 5], np.int32))
    assert res["num_accepted"].tolist() == [2, 0, 5]
    assert res["out_tokens"][0].tolist() == [x[0, 0], x[0, 1], am[0, 2], -1, -1, -1]
    assert res["out_tokens"][1].tolist() == [am[1, 0], -1, -1, -1, -1, -1]
    assert res["out_tokens"][2].tolist() == x[2].tolist() + [am[2, 5]]


def test_width_ignores_rows_past_it(oracle):
    """A NaN in a row past the width and an invalid proposal past it leave the
    request valid; a width outside [0, gamma] is a bad token (status 5)."""
    V, gamma, B = 16, 4, 4
    rng = np.random.default_rng(26)
    t = rng.normal(0, 1, (B, gamma + 1, V)).astype(np.float32)
    t[0, 3, 5] = np.nan
    x = t.argmax(-1)[:, :gamma].astype(np.int32)
    x[1, 3] = V + 7
    pol = synth.uniform_policy(B, greedy=True).numpy()
    res = oracle.verify(t, x, None, None, pol, **synth.make_keys(B).numpy(),
                        width=np.array([2, 3, gamma + 1, -1], np.int32))
    assert res["status"].tolist() == [0, 0, 5, 5]
    assert res["num_accepted"].tolist()[:2] == [2, 3]


@pytest.mark.parametrize("policy", ["sampled", "greedy"])
def test_width_is_the_truncated_block(oracle, policy):
    """Verifying at width w is the fixed-width verify of the block cut to
    x_1..x_w and target rows 0..w, under the same keys: the accept tests, the
    residual and the bonus draw at the same positions.  The tail past w is -1."""
    V, gamma, B = 64, 4, 96
    rng = np.random.default_rng(27)
    t = rng.normal(0, 2.0, (B, gamma + 1, V)).astype(np.float32)
    d_logits = t[:, :gamma] + rng.normal(0, 1.0, (B, gamma, V))
    q = np.exp(d_logits - d_logits.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    x = np.array([[rng.choice(V, p=q[b, k] / q[b, k].sum()) for k in range(gamma)] for b in range(B)], np.int32)
    qx = np.take_along_axis(q, x[..., None], 2)[..., 0]
    pol = synth.uniform_policy(B, greedy=policy == "greedy").numpy()
    keys = synth.make_keys(B, seed=9, pos0=1000).numpy()
    for w in range(1, gamma + 1):
        res = oracle.verify(t, x, q, qx, pol, **keys, width=np.full(B, w, np.int32))
        cut = oracle.verify(np.ascontiguousarray(t[:, :w + 1]), np.ascontiguousarray(x[:, :w]),
                            np.ascontiguousarray(q[:, :w]), np.ascontiguousarray(qx[:, :w]), pol, **keys)
        np.testing.assert_array_equal(res["status"], cut["status"])
        np.testing.assert_array_equal(res["num_accepted"], cut["num_accepted"])
        np.testing.assert_array_equal(res["out_tokens"][:, :w + 1], cut["out_tokens"])
        assert np.all(res["out_tokens"][:, w + 1:] == -1)
        # the accept tests are live: some requests stop early, some run to w
        if policy == "sampled":
            assert (res["num_accepted"] < w).any() and (res["num_accepted"] == w).any()
