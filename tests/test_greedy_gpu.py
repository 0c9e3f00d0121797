"""GPU parity of the greedy paths against the oracle: bit-exact tokens.

Greedy verify compares every output of every request; greedy drafting without
a Markov bias (r = 0) compares proposals exactly and confidences within the
float tolerance."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

TOL_ABS, TOL_REL = 1e-5, 1e-4


@pytest.fixture(scope="module")
def ds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_dspark_markov_gb300 as ds
    from verify_dspark_markov_gb300 import build
    build.build()
    ds.load()
    return ds


def _oracle_verify_greedy(oracle, target, proposals, keys):
    B = target.shape[0]
    return oracle.verify(synth.host(target), proposals.cpu().numpy(), None, None,
                         synth.uniform_policy(B, greedy=True).numpy(), **keys.numpy())


def _gpu_verify_greedy(ds, target, proposals):
    out, nacc, st = ds.verify(target.cuda(), proposals.cuda().to(torch.int32))
    torch.cuda.synchronize()
    return out.cpu().numpy(), nacc.cpu().numpy(), st.cpu().numpy()


def _check_verify(res, got):
    out, nacc, st = got
    np.testing.assert_array_equal(st, res["status"])
    np.testing.assert_array_equal(nacc, res["num_accepted"])
    np.testing.assert_array_equal(out, res["out_tokens"])


def _draft_argmax(oracle, w):
    """Proposals of a greedy r = 0 draft, from the oracle."""
    res = oracle.markov_sample(synth.host(w.backbone), w.anchor.cpu().numpy(), None, None, None, None,
                               None, synth.uniform_policy(w.B, greedy=True).numpy(), **w.keys.numpy())
    return torch.from_numpy(res["proposals"])


def test_verify_greedy_tiny(ds, oracle):
    w = synth.tiny(greedy=True)
    x = _draft_argmax(oracle, w)
    _check_verify(_oracle_verify_greedy(oracle, w.target, x, w.keys), _gpu_verify_greedy(ds, w.target, x))


def test_verify_greedy_full_decode_tile(ds, oracle):
    """The 64-request x 8-row, 129,280-vocabulary bf16 tile with planted exact
    ties, in the launch configuration the benchmark times."""
    w = synth.full_decode_tile(device="cuda")
    x = _draft_argmax(oracle, w)
    res = _oracle_verify_greedy(oracle, w.target, x, w.keys)
    _check_verify(res, _gpu_verify_greedy(ds, w.target, x))
    assert (res["num_accepted"] < w.gamma).any()


@pytest.mark.parametrize("B,gamma,V,dtype", [
    (1, 1, 8, torch.float32), (3, 16, 8, torch.bfloat16), (5, 3, 1032, torch.bfloat16),
    (7, 4, 40_008, torch.float32), (33, 2, 4096, torch.bfloat16), (2, 5, 262_144, torch.bfloat16),
    (300, 1, 64, torch.float32)])
def test_verify_greedy_shapes(ds, oracle, B, gamma, V, dtype):
    """Ragged splits: rows smaller than one CTA's range, rows spanning many
    CTAs, a vocabulary that is not a multiple of the vector tiles."""
    g = torch.Generator().manual_seed(B * 1000 + V)
    t = torch.randint(-4, 5, (B, gamma + 1, V), generator=g).to(torch.float32) / 2  # many exact ties
    t = t.to(dtype)
    a = t.float().argmax(dim=2)
    x = torch.where(torch.rand((B, gamma), generator=g) < 0.7, a[:, :gamma],
                    torch.randint(0, V, (B, gamma), generator=g)).to(torch.int32)
    keys = synth.make_keys(B)
    _check_verify(_oracle_verify_greedy(oracle, t, x, keys), _gpu_verify_greedy(ds, t, x))


def test_verify_greedy_special_values(ds, oracle):
    B, gamma, V = 6, 3, 256
    t = torch.randn((B, gamma + 1, V), generator=torch.Generator().manual_seed(3))
    t[0, 2, 17] = float("nan")                   # non-finite
    t[1, 0, 3] = float("inf")                    # non-finite
    t[2, 1, :] = float("-inf")                   # empty row
    t[3, :, :] = 0.0                             # -0 / +0 ties resolve to the lowest index
    t[3, :, 0] = -0.0
    t[4, 3, 200:] = float("-inf")
    x = t.argmax(dim=2)[:, :gamma].to(torch.int32)
    x[5, 1] = V                                  # proposal out of range
    x[3, 0] = 0
    keys = synth.make_keys(B)
    res = _oracle_verify_greedy(oracle, t, x, keys)
    got = _gpu_verify_greedy(ds, t, x)
    _check_verify(res, got)
    assert res["status"].tolist() == [1, 1, 2, 0, 0, 5]


def test_verify_greedy_needs_no_workspace_and_repeats(ds, oracle):
    """The greedy verify keeps its state on chip: repeated calls give the same
    result and the binding never allocates a workspace for them."""
    w = synth.full_decode_tile(V=8192, B=16, device="cuda")
    x = _draft_argmax(oracle, w).cuda()
    wsp = ds.Workspace()
    first = ds.verify(w.target, x, workspace=wsp)
    for _ in range(3):
        again = ds.verify(w.target, x, workspace=wsp)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    assert wsp._bufs == {}


def test_draft_greedy_r0_with_confidence(ds, oracle):
    w = synth.tiny(greedy=True, r=0, H=64)
    E = w.weights.E
    res = oracle.markov_sample(synth.host(w.backbone), w.anchor.numpy(), None, None, synth.host(w.h),
                               synth.host(E), w.weights.w_conf.numpy(), w.policy.numpy(), **w.keys.numpy())
    got = ds.markov_sample(w.backbone.cuda(), w.anchor.cuda(), h=w.h.cuda(), E=E.cuda(),
                           w_conf=w.weights.w_conf.cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got["status"].cpu().numpy(), res["status"])
    np.testing.assert_array_equal(got["proposals"].cpu().numpy(), res["proposals"])
    np.testing.assert_array_equal(got["q_at_x"].cpu().numpy(), res["q_at_x"])
    np.testing.assert_allclose(got["conf"].cpu().numpy(), res["conf"], atol=TOL_ABS, rtol=TOL_REL)


def test_draft_greedy_r0_full_decode_tile(ds, oracle):
    w = synth.full_decode_tile(device="cuda")
    res = oracle.markov_sample(synth.host(w.backbone), w.anchor.cpu().numpy(), None, None, None, None,
                               None, synth.uniform_policy(w.B, greedy=True).numpy(), **w.keys.numpy())
    got = ds.markov_sample(w.backbone, w.anchor)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got["proposals"].cpu().numpy(), res["proposals"])
    np.testing.assert_array_equal(got["status"].cpu().numpy(), res["status"])


def test_draft_greedy_bad_anchor_and_nan(ds, oracle):
    B, gamma, V = 3, 4, 64
    bb = torch.randn((B, gamma, V), generator=torch.Generator().manual_seed(9))
    bb[2, 2, 5] = float("nan")
    anchor = torch.tensor([1, V, 3], dtype=torch.int32)
    H = 8
    h = torch.randn((B, gamma, H))
    E = torch.randn((V, H)).to(torch.bfloat16)
    wc = torch.randn(2 * H)
    res = oracle.markov_sample(bb.numpy(), anchor.numpy(), None, None, h.numpy(), synth.host(E),
                               wc.numpy(), synth.uniform_policy(B, greedy=True).numpy(),
                               **synth.make_keys(B).numpy())
    got = ds.markov_sample(bb.cuda(), anchor.cuda(), h=h.cuda(), E=E.cuda(), w_conf=wc.cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got["status"].cpu().numpy(), res["status"])
    np.testing.assert_array_equal(got["proposals"].cpu().numpy(), res["proposals"])
    np.testing.assert_array_equal(got["q_at_x"].cpu().numpy(), res["q_at_x"])
    np.testing.assert_allclose(got["conf"].cpu().numpy(), res["conf"], atol=TOL_ABS, rtol=TOL_REL)
