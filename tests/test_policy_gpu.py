"""GPU parity of the sampled paths (per-request temperature / top-k / top-p):
dspark_verify with policies and dspark_markov_sample with policies.

Tokens and decisions are compared exactly wherever the oracle marks them
determinate (outside the 1e-5 bands around an accept threshold, an inverse-CDF
boundary, a top-p cut or a near-tie of rounded logits); indeterminate cases
are counted, and after the first one a request's later outputs are not
compared.  Probabilities agree within 1e-5 absolute / 1e-4 relative."""
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


def _keys_dev(keys):
    return dict(seed=keys.seed.cuda(), request_id=keys.request_id.cuda(), pos0=keys.pos0.cuda())


def _draft_oracle(oracle, w, with_h=False):
    return oracle.markov_sample(synth.host(w.backbone), w.anchor.cpu().numpy(), None, None,
                                synth.host(w.h) if with_h else None,
                                synth.host(w.weights.E) if with_h else None,
                                w.weights.w_conf.cpu().numpy() if with_h else None,
                                w.policy.numpy(), **w.keys.numpy())


def _verify_both(ds, oracle, w, draft):
    ref = oracle.verify(synth.host(w.target), draft["proposals"], draft["q"], draft["q_at_x"],
                        w.policy.numpy(), **w.keys.numpy())
    dev = w.target.device if w.target.is_cuda else torch.device("cuda")
    out, nacc, st = ds.verify(w.target.to(dev), torch.from_numpy(draft["proposals"]).to(dev),
                              q=torch.from_numpy(draft["q"]).to(dev),
                              q_at_x=torch.from_numpy(draft["q_at_x"]).to(dev),
                              policy=w.policy.packed().to(dev), **_keys_dev(w.keys))
    torch.cuda.synchronize()
    return ref, (out.cpu().numpy(), nacc.cpu().numpy(), st.cpu().numpy())


def _check_verify(ref, got, max_indet_frac=0.05):
    """Status of every request; every output of a determinate request; of an
    indeterminate one, the tokens emitted before its first indeterminate
    decision (and num_accepted when it was decided before it).  Returns the
    number of indeterminate requests."""
    out, nacc, st = got
    np.testing.assert_array_equal(st, ref["status"])
    det = ~ref["indet"]
    assert det.mean() >= 1 - max_indet_frac, f"{(~det).sum()} indeterminate of {det.size}"
    np.testing.assert_array_equal(nacc[det], ref["num_accepted"][det])
    np.testing.assert_array_equal(out[det], ref["out_tokens"][det])
    partial = 0
    for b in np.flatnonzero(~det):
        n = int(ref["det_tokens"][b])
        np.testing.assert_array_equal(out[b, :n], ref["out_tokens"][b, :n], err_msg=f"request {b}")
        partial += n
        if ref["det_nacc"][b]:
            assert nacc[b] == ref["num_accepted"][b], b
    if (~det).any():
        print(f"indeterminate requests: {(~det).sum()} of {det.size}; "
              f"{partial} tokens of theirs compared before the first indeterminate decision")
    return int((~det).sum())


def _check_draft(ref, got, V, max_indet_frac=0.05):
    np.testing.assert_array_equal(got["status"].cpu().numpy(), ref["status"])
    props = got["proposals"].cpu().numpy()
    qx = got["q_at_x"].cpu().numpy()
    q = None if got["q"] is None else got["q"].cpu().numpy()
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
    assert indet <= max(1, max_indet_frac * B * gamma)
    return indet


# ----------------------------------------------------------------- verify
def test_verify_sampled_tiny(ds, oracle):
    w = synth.tiny(r=0, H=0)
    draft = _draft_oracle(oracle, w)
    _check_verify(*_verify_both(ds, oracle, w, draft))


@pytest.mark.parametrize("V,B", [(4096, 24), (129_280, 64)])
def test_verify_sampled_decode_tile(ds, oracle, V, B):
    """T = 0.7, top-k 50, top-p 0.95 on Zipf-shaped bf16 rows (the full-size
    case is the 64-request, gamma = 5 decode verify tile)."""
    w = synth.decode_verify_tile(V=V, B=B, r=0, H=0, device="cuda" if V > 10000 else "cpu")
    draft = _draft_oracle(oracle, w)
    _check_verify(*_verify_both(ds, oracle, w, draft))


@pytest.mark.parametrize("V,B,indet", [(8192, 96, 0.05), (129_280, 40, 0.35)])
def test_verify_sampled_mixed_policies(ds, oracle, V, B, indet):
    """Per-request T, top-k in {0, 20, 100, 1000}, top-p in {1, 0.9, 0.8},
    25 % greedy, 10 % adversarial drafts.  At full vocabulary a token near a
    top-p cut holds ~1e-4 of the mass, so the 1e-5 band around p marks about
    one row in five indeterminate."""
    w = synth.mixed_serving(V=V, B=B, r=0, H=0, adversarial_frac=0.1)
    draft = _draft_oracle(oracle, w)
    n = _check_verify(*_verify_both(ds, oracle, w, draft), max_indet_frac=indet)
    print(f"indeterminate requests: {n} of {B}")


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_verify_sampled_flat_rows(ds, oracle, dtype):
    """Flat rows (N(0, 0.5) logits, V = 129,280): top-p cuts inside steps of
    thousands of tokens (in bf16, ties hundreds deep), top-k of 5,000 and
    20,000 with and without top-p, and a row without truncation."""
    w = synth.flat_rows(B=48, dtype=dtype)
    draft = _draft_oracle(oracle, w)
    # ~1e-4 of the mass per token near every cut and draw boundary: the 1e-5
    # bands mark most requests indeterminate (the drafting test below compares
    # the same row engine's full q rows)
    n = _check_verify(*_verify_both(ds, oracle, w, draft), max_indet_frac=0.85)
    print(f"indeterminate requests: {n} of {w.B}")


def test_verify_sampled_special_cases(ds, oracle):
    w = synth.decode_verify_tile(V=1024, B=6, r=0, H=0, sigmas=(2.0,))
    draft = _draft_oracle(oracle, w)                   # drafted under the original policies
    w.policy.temperature[1] = 0.0                      # invalid verify policy
    w.policy.top_k[2] = 1                              # top-k 1: one-hot
    w.policy.top_p[3] = 1e-7                           # top-p -> 0: one-hot
    w.policy.greedy[4] = 1                             # a greedy request in the batch
    w.target[5, 3, 11] = float("nan")                  # non-finite row
    ref, got = _verify_both(ds, oracle, w, draft)
    assert ref["status"].tolist()[1] == 4 and ref["status"].tolist()[5] == 1
    _check_verify(ref, got, max_indet_frac=0.34)


def test_verify_sampled_preserves_target_law(ds):
    """The emitted-token law equals target-only sampling on a tiny vocabulary
    (chi-square, alpha = 1e-3): first token ~ p_0, second (given x_1
    accepted) ~ p_1, for agreeing / disagreeing / nearly disjoint drafts."""
    from scipy import stats
    V, gamma, B = 8, 3, 200_000
    rng = np.random.default_rng(31)
    for regime in ("agreeing", "disagreeing", "nearly_disjoint"):
        t_logits = rng.normal(0, 1.5, (gamma + 1, V))
        if regime == "agreeing":
            d_logits = t_logits[:gamma] + rng.normal(0, 0.3, (gamma, V))
        elif regime == "disagreeing":
            d_logits = rng.normal(0, 1.5, (gamma, V))
        else:
            t_logits[:, 4:] = -np.inf
            d_logits = np.zeros((gamma, V))
            d_logits[:, :4] = -6.0
        p_rows = torch.softmax(torch.tensor(t_logits), -1).numpy()
        q_rows = torch.softmax(torch.tensor(d_logits), -1).numpy()
        x = np.stack([rng.choice(V, size=B, p=q_rows[k]) for k in range(gamma)], 1).astype(np.int32)
        t = torch.tensor(t_logits, dtype=torch.float32).expand(B, gamma + 1, V).contiguous().cuda()
        q = torch.tensor(q_rows, dtype=torch.float32).expand(B, gamma, V).contiguous().cuda()
        xd = torch.from_numpy(x).cuda()
        qx = torch.gather(q, 2, xd.long()[..., None])[..., 0].contiguous()
        pol = synth.uniform_policy(B, temperature=1.0).packed().cuda()
        keys = synth.make_keys(B, seed=7)
        out, nacc, st = ds.verify(t, xd, q=q, q_at_x=qx, policy=pol, **_keys_dev(keys))
        out, nacc = out.cpu().numpy(), nacc.cpu().numpy()
        assert np.all(st.cpu().numpy() == 0)
        for tokens, p in ((out[:, 0], p_rows[0]), (out[nacc >= 1, 1], p_rows[1])):
            if len(tokens) < 2000:
                continue
            sup = p > 0
            assert np.all(sup[tokens])
            c = np.bincount(tokens, minlength=V)[sup]
            assert stats.chisquare(c, p[sup] * c.sum()).pvalue > 1e-3, regime


# ----------------------------------------------------------------- draft
def test_draft_sampled_tiny(ds, oracle):
    w = synth.tiny(r=0, H=64)
    ref = _draft_oracle(oracle, w, with_h=True)
    got = ds.markov_sample(w.backbone.cuda(), w.anchor.cuda(), h=w.h.cuda(), E=w.weights.E.cuda(),
                           w_conf=w.weights.w_conf.cuda(), policy=w.policy.packed().cuda(),
                           **_keys_dev(w.keys))
    torch.cuda.synchronize()
    _check_draft(ref, got, w.V)
    np.testing.assert_allclose(got["conf"].cpu().numpy(), ref["conf"], atol=ATOL, rtol=RTOL)


@pytest.mark.parametrize("maker,kw", [
    (synth.decode_verify_tile, dict(V=4096, B=16)),
    (synth.mixed_serving, dict(V=8192, B=64)),
    (synth.decode_verify_tile, dict(V=129_280, B=64, device="cuda"))])
def test_draft_sampled_policies(ds, oracle, maker, kw):
    w = maker(r=0, H=0, **kw)
    ref = _draft_oracle(oracle, w)
    dev = torch.device("cuda")
    got = ds.markov_sample(w.backbone.to(dev), w.anchor.to(dev), policy=w.policy.packed().to(dev),
                           **_keys_dev(w.keys))
    torch.cuda.synchronize()
    _check_draft(ref, got, w.V)


def test_draft_sampled_mixed_full_vocab(ds, oracle):
    """Mixed policies at V = 129,280: rows with top-k 1,000 and top-p cut
    inside the top-k set leave a gap of whole bins between the two cuts."""
    w = synth.mixed_serving(V=129_280, B=32, r=0, H=0, device="cuda")
    ref = _draft_oracle(oracle, w)
    got = ds.markov_sample(w.backbone, w.anchor, policy=w.policy.packed(), **_keys_dev(w.keys))
    torch.cuda.synchronize()
    n = _check_draft(ref, got, w.V, max_indet_frac=0.35)
    print(f"indeterminate positions: {n} of {w.B * w.gamma}")


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_draft_sampled_flat_rows(ds, oracle, dtype):
    """Drafting on flat rows, bf16 and fp32 (fp32 rows take the same row
    engine as the Markov logits; with the bias on, logits this dense sit
    within the rounding band of every cut, which the oracle marks
    indeterminate)."""
    w = synth.flat_rows(B=24, dtype=dtype)
    ref = _draft_oracle(oracle, w)
    got = ds.markov_sample(w.backbone.cuda(), w.anchor.cuda(), policy=w.policy.packed().cuda(),
                           **_keys_dev(w.keys))
    torch.cuda.synchronize()
    n = _check_draft(ref, got, w.V, max_indet_frac=0.5)
    print(f"indeterminate positions: {n} of {w.B * w.gamma}")


def test_workspace_reuse_across_sizes(ds, oracle):
    """One workspace shared by calls of different sizes and paths, in turn
    (sampled verify, greedy verify, Markov drafting with and without the
    bias): every call must find its counters at zero and match the oracle."""
    wsp = ds.Workspace()
    for (V, B, r) in ((2048, 24, 0), (1024, 5, 64), (4096, 40, 0), (2048, 3, 16)):
        w = synth.decode_verify_tile(V=V, B=B, r=r, H=0)
        draft = _draft_oracle(oracle, w) if r == 0 else None
        if draft is not None:
            ref = oracle.verify(synth.host(w.target), draft["proposals"], draft["q"], draft["q_at_x"],
                                w.policy.numpy(), **w.keys.numpy())
            got = ds.verify(w.target.cuda(), torch.from_numpy(draft["proposals"]).cuda(),
                            q=torch.from_numpy(draft["q"]).cuda(), q_at_x=torch.from_numpy(draft["q_at_x"]).cuda(),
                            policy=w.policy.packed().cuda(), workspace=wsp, **_keys_dev(w.keys))
            torch.cuda.synchronize()
            _check_verify(ref, tuple(t.cpu().numpy() for t in got))
            x = torch.from_numpy(draft["proposals"]).cuda()
            gref = oracle.verify(synth.host(w.target), draft["proposals"], None, None,
                                 synth.uniform_policy(B, greedy=True).numpy(), **w.keys.numpy())
            ggot = ds.verify(w.target.cuda(), x, workspace=wsp)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(ggot[0].cpu().numpy(), gref["out_tokens"])
        kw = {} if r == 0 else dict(U=w.weights.U.cuda(), W=w.weights.W.cuda())
        mref = oracle.markov_sample(synth.host(w.backbone), w.anchor.numpy(),
                                    synth.host(w.weights.U) if r else None, synth.host(w.weights.W) if r else None,
                                    None, None, None, w.policy.numpy(), **w.keys.numpy())
        mgot = ds.markov_sample(w.backbone.cuda(), w.anchor.cuda(), policy=w.policy.packed().cuda(),
                                workspace=wsp, **kw, **_keys_dev(w.keys))
        torch.cuda.synchronize()
        _check_draft(mref, mgot, V)
