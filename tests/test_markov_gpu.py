"""GPU parity of dspark_markov_sample with the low-rank Markov bias (r > 0,
tensor-core GEMM) against the oracle.

Proposals are compared exactly where the oracle marks the step determinate
(its rounded logits are not within 1e-5 of a tie or cut, and the draw is not
within 1e-5 of a boundary); q, q(x) and the confidences within 1e-5 absolute /
1e-4 relative."""
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


def _both(ds, oracle, w, with_policy=True, with_h=True):
    pol_np = w.policy.numpy() if with_policy else synth.uniform_policy(w.B, greedy=True).numpy()
    ref = oracle.markov_sample(synth.host(w.backbone), w.anchor.cpu().numpy(), synth.host(w.weights.U),
                               synth.host(w.weights.W), synth.host(w.h) if with_h else None,
                               synth.host(w.weights.E) if with_h else None,
                               w.weights.w_conf.cpu().numpy() if with_h else None, pol_np, **w.keys.numpy())
    dev = torch.device("cuda")
    keys = dict(seed=w.keys.seed.to(dev), request_id=w.keys.request_id.to(dev), pos0=w.keys.pos0.to(dev))
    got = ds.markov_sample(w.backbone.to(dev), w.anchor.to(dev), U=w.weights.U.to(dev), W=w.weights.W.to(dev),
                           h=w.h.to(dev) if with_h else None, E=w.weights.E.to(dev) if with_h else None,
                           w_conf=w.weights.w_conf.to(dev) if with_h else None,
                           policy=w.policy.packed().to(dev) if with_policy else None, **keys)
    torch.cuda.synchronize()
    return ref, got


def _check(ref, got, max_indet_frac=0.05, with_h=True):
    np.testing.assert_array_equal(got["status"].cpu().numpy(), ref["status"])
    props = got["proposals"].cpu().numpy()
    qx = got["q_at_x"].cpu().numpy()
    q = None if got["q"] is None else got["q"].cpu().numpy()
    conf = got["conf"].cpu().numpy() if with_h else None
    B, gamma = props.shape
    indet = 0
    for b in range(B):
        for k in range(gamma):
            if with_h:  # c_k depends on x_{k-1}, which matched so far
                np.testing.assert_allclose(conf[b, k], ref["conf"][b, k], atol=ATOL, rtol=RTOL)
            if ref["indet"][b, k]:
                indet += 1
                break
            assert props[b, k] == ref["proposals"][b, k], (b, k)
            np.testing.assert_allclose(qx[b, k], ref["q_at_x"][b, k], atol=ATOL, rtol=RTOL)
            if q is not None and not np.all(ref["q"][b, k] == 0):
                np.testing.assert_allclose(q[b, k], ref["q"][b, k], atol=ATOL, rtol=RTOL)
    assert indet <= max(1, max_indet_frac * B * gamma), indet
    return indet


@pytest.mark.parametrize("greedy", [False, True])
def test_markov_tiny_rank16(ds, oracle, greedy):
    """Configuration-1 recipe: V = 1024, r = 16 (a single MMA K step), H = 64,
    T = 1 without truncation, or greedy."""
    w = synth.tiny(r=16, H=64, greedy=greedy)
    ref, got = _both(ds, oracle, w)
    _check(ref, got)


@pytest.mark.parametrize("B,V,r", [(5, 4096, 256), (16, 4096, 64), (33, 2056, 128), (160, 2056, 256),
                                   (200, 1032, 48), (129, 1000, 16), (1, 50000, 192), (48, 50000, 64),
                                   (8, 150000, 128)])
def test_markov_ragged_batches(ds, oracle, B, V, r):
    """Batches that do not fill the 128-request M tile (padding rows) or need
    two of them (B > 128), vocabularies that are not a multiple of the
    vocabulary tile, and ranks that are not a multiple of 64 (the W tiles then
    arrive without swizzle).  Up to 64 requests with r a multiple of 64 run
    the fused draft: V = 50,000 gives each CTA three vocabulary tiles and a
    ragged last tile, V = 150,000 eight tiles (all of tensor memory) and a
    ragged last tile."""
    w = synth.decode_verify_tile(V=V, B=B, r=r, H=32)
    ref, got = _both(ds, oracle, w)
    _check(ref, got)


def test_markov_mixed_policies_rank256(ds, oracle):
    w = synth.mixed_serving(V=8192, B=64, r=256, H=64)
    ref, got = _both(ds, oracle, w)
    _check(ref, got)


def test_markov_nonfinite_rows_rank64(ds, oracle):
    """Rows the bias kernel's maxima must flag: NaN at step 1, +inf at step 3,
    every logit -inf at step 2 (no maximum) - each in its own request."""
    w = synth.decode_verify_tile(V=4096, B=8, r=64, H=0)
    bb = w.backbone.float()
    bb[1, 0, 17] = float("nan")
    bb[2, 2, 5] = float("inf")
    bb[3, 1, :] = float("-inf")
    w.backbone = bb.to(w.backbone.dtype).contiguous()
    ref, got = _both(ds, oracle, w, with_h=False)
    assert ref["status"].tolist()[1:4] == [1, 1, 2], ref["status"]
    _check(ref, got, with_h=False, max_indet_frac=0.25)


def test_markov_greedy_no_policy(ds, oracle):
    w = synth.decode_verify_tile(V=4096, B=24, r=256, H=0)
    ref, got = _both(ds, oracle, w, with_policy=False, with_h=False)
    _check(ref, got, with_h=False)


def test_markov_full_vocab_rank256(ds, oracle):
    """The decode verify tile's draft at full vocabulary and rank (16 of its
    64 requests, which the oracle computes in a few seconds)."""
    w = synth.decode_verify_tile(B=16, H=4096, device="cuda")
    ref, got = _both(ds, oracle, w)
    _check(ref, got)



@pytest.mark.parametrize("B,V,r", [(5, 4096, 256), (33, 2056, 128), (160, 2056, 64)])
def test_markov_fp32_backbone(ds, oracle, B, V, r):
    """The bias GEMM's fp32-backbone epilogue, which no bf16 case reaches (the
    RNN-head draft's second product runs on it): fp32 backbone rows at three
    ranks and ragged batches."""
    w = synth.decode_verify_tile(V=V, B=B, r=r, H=0, seed=3001 + B)
    w.backbone = w.backbone.float().contiguous()
    ref, got = _both(ds, oracle, w, with_h=False)
    _check(ref, got, with_h=False)
