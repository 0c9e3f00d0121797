"""Pins of the oracle's RNN-head sampler (a GRU state carried across the
block, its low-rank bias added to the backbone logits).  The pages name the
head without equations, so these pins tie the oracle to the GRU cell's
textbook definition (a float64 library GRU cell), to the backbone-only
sampler and to closed forms, not to printed values."""
import numpy as np
import pytest
import torch

import synth

V, R, GAMMA, B = 64, 16, 5, 12


def _bf16(a):
    return synth.bf16_bits(torch.tensor(a, dtype=torch.float32).to(torch.bfloat16))


def _f64(bits):
    return synth.from_bf16_bits(bits).double().numpy()


def _weights(seed, scale=0.4):
    rng = np.random.default_rng(seed)
    return dict(U=_bf16(rng.normal(0, 1.0, (V, R))), W=_bf16(rng.normal(0, 0.5, (V, R))),
                Wi=_bf16(rng.normal(0, scale, (3 * R, R))), Wh=_bf16(rng.normal(0, scale, (3 * R, R))),
                bi=rng.normal(0, 0.3, 3 * R).astype(np.float32), bh=rng.normal(0, 0.3, 3 * R).astype(np.float32))


def _run(oracle, wts, seed=5, policy=None):
    rng = np.random.default_rng(seed)
    backbone = rng.normal(0, 2.0, (B, GAMMA, V)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    pol = (policy or synth.uniform_policy(B)).numpy()
    res = oracle.rnn_sample(backbone, anchor, wts["U"], wts["W"], wts["Wi"], wts["Wh"], wts["bi"], wts["bh"],
                            None, None, None, pol, **synth.make_keys(B, seed=seed).numpy())
    return backbone, anchor, res


def _library_states(wts, anchor, proposals):
    """s_k of a float64 torch GRU cell fed U[x_{k-1}], from s_0 = 0."""
    cell = torch.nn.GRUCell(R, R, dtype=torch.float64)
    with torch.no_grad():
        cell.weight_ih.copy_(torch.from_numpy(_f64(wts["Wi"])))
        cell.weight_hh.copy_(torch.from_numpy(_f64(wts["Wh"])))
        cell.bias_ih.copy_(torch.from_numpy(wts["bi"].astype(np.float64)))
        cell.bias_hh.copy_(torch.from_numpy(wts["bh"].astype(np.float64)))
        U = torch.from_numpy(_f64(wts["U"]))
        s = torch.zeros((B, R), dtype=torch.float64)
        out = []
        prev = torch.from_numpy(anchor.astype(np.int64))
        for k in range(GAMMA):
            s = cell(U[prev], s)
            out.append(s.numpy().copy())
            prev = torch.from_numpy(proposals[:, k].astype(np.int64))
    return np.stack(out, 1)


def test_rnn_states_are_a_library_gru_cell(oracle):
    wts = _weights(41)
    _, anchor, res = _run(oracle, wts)
    assert np.all(res["status"] == 0)
    ref = _library_states(wts, anchor, res["proposals"])
    np.testing.assert_allclose(res["states"], ref, rtol=0, atol=1e-12)
    assert np.abs(ref).max() > 0.1  # the state is far from zero


def test_rnn_q_follows_the_state_bias(oracle):
    """T = 1, no truncation: log q_k differs from the fp32-rounded logits
    backbone + W s_k (the library states) by a constant per row."""
    wts = _weights(42)
    backbone, anchor, res = _run(oracle, wts, seed=6)
    s = _library_states(wts, anchor, res["proposals"])
    z = (backbone.astype(np.float64) + np.einsum("bkj,vj->bkv", s, _f64(wts["W"]))).astype(np.float32)
    z = z.astype(np.float64)
    lq = np.log(res["q"].astype(np.float64))
    np.testing.assert_allclose(lq - lq[..., :1], z - z[..., :1], rtol=0, atol=2e-6)
    # the bias is not negligible, and it changes from step to step
    bias = z - backbone
    assert np.abs(bias).max() > 0.5 and np.abs(np.diff(bias, axis=1)).max() > 0.1


def test_rnn_update_gate_at_one_is_backbone_only(oracle):
    """An update gate held at 1 keeps s_k = s_0 = 0: no bias, so the proposals,
    q and q(x) are those of the sampler without a head (rank 0)."""
    wts = _weights(43)
    wts["bi"][R:2 * R] = 60.0  # sigma(60) rounds to 1 in double
    pol = synth.Policy(torch.full((B,), 0.8), torch.tensor([0, 5, 20] * (B // 3), dtype=torch.int32),
                       torch.full((B,), 0.9), torch.tensor([0, 0, 0, 1] * (B // 4), dtype=torch.int32))
    backbone, anchor, res = _run(oracle, wts, seed=7, policy=pol)
    assert np.all(res["states"] == 0.0)
    ref = oracle.markov_sample(backbone, anchor, None, None, None, None, None, pol.numpy(),
                               **synth.make_keys(B, seed=7).numpy())
    for k in ("proposals", "q", "q_at_x", "status"):
        np.testing.assert_array_equal(res[k], ref[k])


def test_rnn_without_carry_is_a_token_function(oracle):
    """Update gate at 0 and no hidden weights: s_k = tanh(Wi_n U[x_{k-1}] +
    bi_n), a function of the previous token alone."""
    wts = _weights(44)
    wts["bi"][R:2 * R] = -60.0
    wts["Wh"][:] = 0
    wts["bh"][:] = 0.0
    _, anchor, res = _run(oracle, wts, seed=8)
    prev = np.concatenate([anchor[:, None], res["proposals"][:, :-1]], 1)
    Win = _f64(wts["Wi"])[2 * R:]
    want = np.tanh(np.einsum("gj,bkj->bkg", Win, _f64(wts["U"])[prev]) + wts["bi"][2 * R:].astype(np.float64))
    np.testing.assert_allclose(res["states"], want, rtol=0, atol=1e-12)


def test_rnn_bad_anchor(oracle):
    wts = _weights(45)
    rng = np.random.default_rng(9)
    backbone = rng.normal(0, 1.0, (B, GAMMA, V)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    anchor[3] = V
    res = oracle.rnn_sample(backbone, anchor, wts["U"], wts["W"], wts["Wi"], wts["Wh"], wts["bi"], wts["bh"],
                            None, None, None, synth.uniform_policy(B).numpy(), **synth.make_keys(B).numpy())
    assert res["status"][3] == 5 and np.all(res["proposals"][3] == -1)
    assert np.all(np.delete(res["status"], 3) == 0)


def test_rnn_confidence_is_the_markov_heads(oracle):
    """The confidence c_k = sigmoid(w^T [h_k ; E[x_{k-1}]]) is the sampler's,
    not the head's: with the update gate at one (no bias) the RNN sampler's
    proposals and confidences equal the backbone-only sampler's."""
    wts = _weights(46)
    wts["bi"][R:2 * R] = 60.0
    rng = np.random.default_rng(10)
    H = 8
    backbone = rng.normal(0, 2.0, (B, GAMMA, V)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    h = rng.normal(0, 1.0, (B, GAMMA, H)).astype(np.float32)
    E = _bf16(rng.normal(0, 1.0, (V, H)))
    w_conf = rng.normal(0, 0.5, 2 * H).astype(np.float32)
    pol = synth.uniform_policy(B).numpy()
    keys = synth.make_keys(B, seed=11).numpy()
    res = oracle.rnn_sample(backbone, anchor, wts["U"], wts["W"], wts["Wi"], wts["Wh"], wts["bi"], wts["bh"],
                            h, E, w_conf, pol, **keys)
    ref = oracle.markov_sample(backbone, anchor, None, None, h, E, w_conf, pol, **keys)
    np.testing.assert_array_equal(res["proposals"], ref["proposals"])
    np.testing.assert_array_equal(res["conf"], ref["conf"])
    # and it uses x_{k-1}: the first position's confidence reads the anchor's E row
    e0 = _f64(E)[anchor]
    want = 1.0 / (1.0 + np.exp(-(h[:, 0].astype(np.float64) @ w_conf[:H] + e0 @ w_conf[H:])))
    np.testing.assert_allclose(res["conf"][:, 0], want, rtol=1e-6)
