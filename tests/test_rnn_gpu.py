"""GPU parity of the RNN-head draft (dspark_rnn_sample) against the oracle:
proposals exact wherever the oracle marks them determinate, q and q(x)
within 1e-5 absolute / 1e-4 relative, confidences within the same.  The
device carries s_k into the logits as a bf16 pair (hi, lo), about 2^-16 of
its size; an emulation of that arithmetic stays within 1e-6 of the exact
state's logits, inside the oracle's 1e-5 indeterminate bands."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
ATOL, RTOL = 1e-5, 1e-4


@pytest.fixture(scope="module")
def ds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_dspark_markov_gb300 as ds
    from verify_dspark_markov_gb300 import build
    build.build()
    ds.load()
    return ds


def _case(V, B, r, H, seed, greedy=False):
    w = synth.decode_verify_tile(V=V, B=B, r=r, H=H, seed=seed)
    gw = synth.gru_weights(r, synth._gen(seed + 1, "cpu"), "cpu")
    if greedy:
        w.policy = synth.uniform_policy(B, greedy=True)
    return w, gw


def _both(ds, oracle, w, gw, policy=True):
    ref = oracle.rnn_sample(synth.host(w.backbone), w.anchor.cpu().numpy(), synth.host(w.weights.U),
                            synth.host(w.weights.W), synth.host(gw.Wi), synth.host(gw.Wh), gw.bi.numpy(),
                            gw.bh.numpy(), synth.host(w.h) if w.h is not None else None,
                            synth.host(w.weights.E) if w.h is not None else None,
                            w.weights.w_conf.cpu().numpy() if w.h is not None else None,
                            w.policy.numpy(), **w.keys.numpy())
    dev = torch.device("cuda")
    kw = dict(policy=w.policy.packed().to(dev), seed=w.keys.seed.to(dev), request_id=w.keys.request_id.to(dev),
              pos0=w.keys.pos0.to(dev)) if policy else {}
    got = ds.rnn_sample(w.backbone.to(dev), w.anchor.to(dev), w.weights.U.to(dev), w.weights.W.to(dev),
                        gw.Wi.to(dev), gw.Wh.to(dev), gw.bi.to(dev), gw.bh.to(dev),
                        h=w.h.to(dev) if w.h is not None else None,
                        E=w.weights.E.to(dev) if w.h is not None else None,
                        w_conf=w.weights.w_conf.to(dev) if w.h is not None else None, **kw)
    torch.cuda.synchronize()
    return ref, {k: (v.cpu() if v is not None else None) for k, v in got.items()}


def _check(ref, got, max_indet_frac=0.05):
    np.testing.assert_array_equal(got["status"].numpy(), ref["status"])
    props, qx = got["proposals"].numpy(), got["q_at_x"].numpy()
    q = None if got["q"] is None else got["q"].numpy()
    B, gamma = props.shape
    indet = 0
    for b in range(B):
        for k in range(gamma):
            if ref["indet"][b, k]:
                indet += 1
                break
            assert props[b, k] == ref["proposals"][b, k], (b, k)
            np.testing.assert_allclose(qx[b, k], ref["q_at_x"][b, k], atol=ATOL, rtol=RTOL)
            if q is not None and ref["proposals"][b, k] >= 0 and not np.all(ref["q"][b, k] == 0):
                np.testing.assert_allclose(q[b, k], ref["q"][b, k], atol=ATOL, rtol=RTOL)
    if got["conf"] is not None:
        np.testing.assert_allclose(got["conf"].numpy(), ref["conf"], atol=ATOL, rtol=RTOL)
    assert indet <= max(1, max_indet_frac * B * gamma)
    return indet


@pytest.mark.parametrize("V,B,r,H", [(4096, 16, 64, 64), (2056, 33, 128, 0), (4096, 200, 256, 0),
                                     (1032, 12, 48, 0), (50000, 40, 192, 0), (4096, 20, 256, 32)])
def test_rnn_sampled(ds, oracle, V, B, r, H):
    """Up to 64 requests with r a multiple of 64 run the whole draft in one
    launch (GRU cell included); 200 requests, or r = 48, take the per-step
    kernels.  V = 50,000 gives the one-launch path three vocabulary tiles per
    CTA and a ragged last tile; r = 256 takes a single W stage."""
    w, gw = _case(V, B, r, H, seed=2001 + B)
    _check(*_both(ds, oracle, w, gw))


def test_rnn_greedy(ds, oracle):
    w, gw = _case(4096, 24, 64, 0, seed=2002, greedy=True)
    _check(*_both(ds, oracle, w, gw, policy=False))


def test_rnn_full_vocab(ds, oracle):
    """The decode tile's draft shape: 64 requests, rank 256, V = 129,280."""
    w, gw = _case(129_280, 64, 256, 0, seed=2003)
    _check(*_both(ds, oracle, w, gw))


def test_rnn_bad_anchor(ds, oracle):
    w, gw = _case(4096, 8, 64, 0, seed=2004)
    w.anchor[3] = 4096
    ref, got = _both(ds, oracle, w, gw)
    assert ref["status"][3] == 5
    _check(ref, got)


def test_rnn_nonfinite_rows(ds, oracle):
    """Rows the one-launch path must flag (8 requests, r = 64): NaN at step 1,
    +inf at step 3, every logit -inf at step 2 (no maximum) - each in its own
    request; the others draft on."""
    w, gw = _case(4096, 8, 64, 0, seed=2005)
    bb = w.backbone.float()
    bb[1, 0, 17] = float("nan")
    bb[2, 2, 5] = float("inf")
    bb[3, 1, :] = float("-inf")
    w.backbone = bb.to(w.backbone.dtype).contiguous()
    ref, got = _both(ds, oracle, w, gw)
    assert ref["status"].tolist()[1:4] == [1, 1, 2], ref["status"]
    _check(ref, got, max_indet_frac=0.25)
