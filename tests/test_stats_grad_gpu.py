"""GPU parity of dspark_accept_stats_grad (the gradient of the statistics'
loss numerators with respect to the draft and confidence logits) against the
oracle.  Gradient entries agree within 1e-7 absolute / 1e-4 relative except
where p_draft and p_target of a token agree to 1e-6 relative: there the sign
in the L1 gradient is decided by rounding, and those tokens are skipped."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
ATOL, RTOL = 1e-7, 1e-4


@pytest.fixture(scope="module")
def ds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_dspark_markov_gb300 as ds
    from verify_dspark_markov_gb300 import build
    build.build()
    ds.load()
    return ds


def _sign_decided(w):
    """Tokens whose sign(p_d - p_t) does not hinge on rounding (exactly equal
    probabilities, e.g. both 0 under a -1e4 logit, give sign 0 on both sides)."""
    d = w.draft.float().double().cpu()
    t = w.target.float().double().cpu()
    pd, pt = torch.softmax(d, -1), torch.softmax(t, -1)
    return (((pd - pt).abs() > 1e-6 * (pd + pt)) | (pd == pt)).numpy()


def _both(ds, oracle, w, scale):
    mask = None if w.mask is None else w.mask
    rd, rc = oracle.accept_stats_backward(synth.host(w.draft), synth.host(w.target), w.labels.cpu().numpy(),
                                          w.conf_logits.cpu().numpy(),
                                          None if mask is None else mask.cpu().numpy(), scale=scale)
    gd, gc = ds.accept_stats_grad(w.draft.cuda(), w.target.cuda(), w.labels.cuda(), w.conf_logits.cuda(),
                                  None if mask is None else mask.cuda(), scale=scale)
    torch.cuda.synchronize()
    return (rd, rc), (gd.cpu().numpy(), gc.cpu().numpy())


def _compare(ref, got, decided):
    rd, rc = ref
    gd, gc = got
    assert np.array_equal(np.isnan(rd), np.isnan(gd))
    ok = decided & ~np.isnan(rd)
    np.testing.assert_allclose(gd[ok], rd[ok], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(gc, rc, atol=1e-6, rtol=RTOL)
    return int((~decided).sum())


@pytest.mark.parametrize("dtype,V,N,gamma,mask", [
    (synth.F32, 1024, 12, 7, False), (synth.BF16, 4096, 9, 5, True), (synth.F32, 8, 5, 3, True),
    (synth.F32, 40_008, 3, 2, True), (synth.BF16, 129_280, 2, 7, False)])
def test_stats_grad_matches_oracle(ds, oracle, dtype, V, N, gamma, mask):
    w = synth.training_stats(V=V, N=N, gamma=gamma, dtype=dtype, disjoint_frac=0.1, with_mask=mask,
                             device="cuda" if V > 10_000 else "cpu")
    ref, got = _both(ds, oracle, w, scale=1.0 / gamma)
    skipped = _compare(ref, got, _sign_decided(w))
    print(f"tokens with an undecided sign: {skipped} of {w.draft.numel()}")


def test_stats_grad_special_positions(ds, oracle):
    """Identical rows (no L1 part), a NaN logit and a label outside [0, V)
    (NaN rows), masked positions (zeros, even where the row is bad)."""
    w = synth.training_stats(V=2048, N=4, gamma=4, dtype=synth.F32, disjoint_frac=0.0, with_mask=False)
    w.target[0, 0] = w.draft[0, 0]
    w.draft[1, 1, 7] = float("nan")
    w.labels[2, 2] = 2048
    w.mask = torch.ones((4, 4), dtype=torch.uint8)
    w.mask[3, :2] = 0
    ref, got = _both(ds, oracle, w, scale=1.0)
    _compare(ref, got, _sign_decided(w) | np.isnan(ref[0]))
    gd = got[0]
    assert np.all(np.isnan(gd[1, 1])) and np.all(np.isnan(gd[2, 2]))
    assert np.all(gd[3, :2] == 0.0) and np.all(got[1][3, :2] == 0.0)
    w.mask[1, 1] = 0
    ref, got = _both(ds, oracle, w, scale=1.0)
    assert np.all(got[0][1, 1] == 0.0) and got[1][1, 1] == 0.0
