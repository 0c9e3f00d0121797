"""GPU parity at the full shapes of the three large workloads, against the
oracle:

* the decode verify tile (64 requests, gamma 5, V = 129,280, bf16, Markov
  rank 256, draft hidden 4096, T 0.7 / top-k 50 / top-p 0.95): the Markov
  draft and the sampled verify of every request run on the GPU; a seeded
  sample of whole requests is recomputed by the oracle;
* the mixed-policy serving batch (256 requests over two 128-request M tiles of
  the bias GEMM, mixed temperature / top-k / top-p, a quarter greedy, a tenth
  adversarial): the same, the sample covering every policy kind and the
  adversarial requests on both M tiles;
* the training statistics (4096 blocks x 7 x 129,280 fp32): every output of
  the GPU against the oracle run over all 28,672 row pairs.

Requests are independent, so the oracle run on a sub-batch (each request with
its own keys) gives exactly that request's outputs in the full batch.  The
draft is compared up to each request's first indeterminate step, the verify
up to its first indeterminate decision (both counted and printed);
probabilities, confidences and losses within 1e-5 absolute / 1e-4 relative.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import synth
from test_policy_gpu import ATOL, RTOL, _check_draft, _check_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_dspark_markov_gb300 as ds
    from verify_dspark_markov_gb300 import build
    build.build()
    ds.load()
    return ds


def _sub_policy(w, idx):
    return {k: v[idx] for k, v in w.policy.numpy().items()}


def _sub_keys(w, idx):
    return {k: v[idx] for k, v in w.keys.numpy().items()}


def _run_and_compare(ds, oracle, w, idx, draft_indet, verify_indet):
    """Draft then verify the whole batch on the GPU; recompute the requests
    idx with the oracle (the draft from the inputs, the verify from the GPU's
    own draft outputs) and compare."""
    got = ds.markov_sample(w.backbone, w.anchor, U=w.weights.U, W=w.weights.W, h=w.h, E=w.weights.E,
                           w_conf=w.weights.w_conf, policy=w.policy.packed(), seed=w.keys.seed,
                           request_id=w.keys.request_id, pos0=w.keys.pos0)
    out, nacc, st = ds.verify(w.target, got["proposals"], q=got["q"], q_at_x=got["q_at_x"],
                              policy=w.policy.packed(), seed=w.keys.seed, request_id=w.keys.request_id,
                              pos0=w.keys.pos0)
    torch.cuda.synchronize()
    it = torch.as_tensor(idx, device=w.backbone.device)
    pol, keys = _sub_policy(w, idx), _sub_keys(w, idx)
    ref = oracle.markov_sample(synth.host(w.backbone[it]), w.anchor[it].cpu().numpy(),
                               synth.host(w.weights.U), synth.host(w.weights.W), synth.host(w.h[it]),
                               synth.host(w.weights.E), w.weights.w_conf.cpu().numpy(), pol, **keys)
    sub = {k: (v[it] if v is not None else None) for k, v in got.items()}
    # the confidence c_k is compared while x_{k-1} matched the oracle's
    conf = sub["conf"].cpu().numpy()
    for i in range(len(idx)):
        for k in range(w.gamma):
            np.testing.assert_allclose(conf[i, k], ref["conf"][i, k], atol=ATOL, rtol=RTOL)
            if ref["indet"][i, k] or ref["proposals"][i, k] != int(sub["proposals"][i, k]):
                break
    n_draft = _check_draft(ref, sub, w.V, max_indet_frac=draft_indet)
    vref = oracle.verify(synth.host(w.target[it]), sub["proposals"].cpu().numpy(), sub["q"].cpu().numpy(),
                         sub["q_at_x"].cpu().numpy(), pol, **keys)
    n_ver = _check_verify(vref, (out[it].cpu().numpy(), nacc[it].cpu().numpy(), st[it].cpu().numpy()),
                          max_indet_frac=verify_indet)
    print(f"{w.name}: {len(idx)} requests compared; indeterminate draft positions {n_draft}, "
          f"indeterminate verify requests {n_ver}")
    # every request of the batch: a valid outcome
    st_all, nacc_all, out_all = st.cpu().numpy(), nacc.cpu().numpy(), out.cpu().numpy()
    assert np.all(st_all == 0)
    for b in range(w.B):
        n = int(nacc_all[b])
        assert 0 <= n <= w.gamma and 0 <= out_all[b, n] < w.V and np.all(out_all[b, n + 1:] == -1)


def test_decode_verify_tile_full(ds, oracle):
    w = synth.decode_verify_tile(device="cuda")
    assert (w.B, w.gamma, w.V, w.weights.r, w.weights.H) == (64, 5, 129_280, 256, 4096)
    rng = np.random.default_rng(2)
    # both ends of the batch and a spread over the three draft-noise levels
    idx = sorted(set([0, 1, 2, w.B - 1] + rng.choice(w.B, 14, replace=False).tolist()))
    _run_and_compare(ds, oracle, w, np.array(idx), draft_indet=0.05, verify_indet=0.25)


def test_mixed_serving_full(ds, oracle):
    w = synth.mixed_serving(device="cuda")
    assert (w.B, w.gamma, w.V, w.weights.r, w.weights.H) == (256, 5, 129_280, 256, 4096)
    pol = w.policy.numpy()
    G, K, P = pol["greedy"] != 0, pol["top_k"] > 0, pol["top_p"] < 1.0
    kinds = {"greedy": G, "untruncated": ~G & ~K & ~P, "top-k only": ~G & K & ~P,
             "top-p only": ~G & ~K & P, "top-k and top-p": ~G & K & P}
    adv = np.zeros(w.B, bool)
    adv[w.extra["adversarial"]] = True
    kinds["adversarial"] = adv
    rng = np.random.default_rng(5)
    idx = set()
    for name, sel in kinds.items():
        for half in (np.arange(w.B) < 128, np.arange(w.B) >= 128):   # both M tiles of the bias GEMM
            cand = np.flatnonzero(sel & half)
            assert len(cand) > 0, (name, "no request of this kind in this half")
            idx.update(rng.choice(cand, min(2, len(cand)), replace=False).tolist())
    idx = np.array(sorted(idx))
    assert len(idx) >= 16
    # at full vocabulary a token near a top-p cut holds ~1e-4 of the mass, so
    # the 1e-5 band around p marks a fair share of the sampled requests
    _run_and_compare(ds, oracle, w, idx, draft_indet=0.35, verify_indet=0.5)


def test_training_stats_full(ds, oracle):
    """Every output over all 28,672 row pairs.  The oracle runs over the
    blocks in chunks copied to the host one at a time (about 2 GB of host
    memory at once), each chunk split over host threads; the numerators are
    summed over the pieces, a different summation order than one call (within
    1e-9 relative of it, well inside the 1e-4 bound)."""
    w = synth.training_stats(device="cuda")
    assert (w.N, w.gamma, w.V) == (4096, 7, 129_280)
    got = ds.accept_stats(w.draft, w.target, w.labels, w.conf_logits)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in got.items()}
    lab, zc = w.labels.cpu().numpy(), w.conf_logits.cpu().numpy()
    nth = max(1, min(32, os.cpu_count() or 1))
    chunk = 256
    parts = []
    with cf.ThreadPoolExecutor(nth) as ex:   # the oracle call releases the GIL
        for c0 in range(0, w.N, chunk):
            c1 = min(w.N, c0 + chunk)
            d, t = synth.host(w.draft[c0:c1]), synth.host(w.target[c0:c1])
            bounds = np.linspace(0, c1 - c0, nth + 1).astype(int)
            def run(i, d=d, t=t, c0=c0, bounds=bounds):
                a, b = bounds[i], bounds[i + 1]
                return oracle.accept_stats(d[a:b], t[a:b], lab[c0 + a:c0 + b], zc[c0 + a:c0 + b])
            parts += [p for p in ex.map(run, range(nth)) if p["l1"].shape[0] > 0]
            del d, t
    del w
    torch.cuda.empty_cache()
    ref = {k: np.concatenate([p[k] for p in parts]) for k in ("l1", "accept", "tau", "status")}
    ref["loss_num"] = np.sum([p["loss_num"] for p in parts], axis=0)
    ref["report"] = np.sum([p["report"] for p in parts], axis=0)
    ref["num_tokens"] = sum(p["num_tokens"] for p in parts)
    np.testing.assert_array_equal(got["status"], ref["status"])
    for k in ("l1", "accept", "tau"):
        np.testing.assert_allclose(got[k], ref[k], atol=ATOL, rtol=RTOL, err_msg=k)
    np.testing.assert_allclose(got["loss_num"], ref["loss_num"], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(got["report"], ref["report"], atol=ATOL, rtol=RTOL)
    assert int(got["num_tokens"][0]) == ref["num_tokens"] == 4096 * 7
