"""GPU parity of dspark_accept_stats against the oracle.

Floating-point outputs must agree within 1e-5 absolute / 1e-4 relative;
statuses and token counts exactly."""
import math

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


def _run(ds, w):
    out = ds.accept_stats(w.draft.cuda(), w.target.cuda(), w.labels.cuda(), w.conf_logits.cuda(),
                          None if w.mask is None else w.mask.cuda())
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _oracle(oracle, w):
    return oracle.accept_stats(synth.host(w.draft), synth.host(w.target), w.labels.cpu().numpy(),
                               w.conf_logits.cpu().numpy(),
                               None if w.mask is None else w.mask.cpu().numpy())


def _compare(got, ref):
    np.testing.assert_allclose(got["l1"], ref["l1"], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(got["accept"], ref["accept"], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(got["tau"], ref["tau"], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(got["loss_num"], ref["loss_num"], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(got["report"], ref["report"], atol=ATOL, rtol=RTOL)
    assert int(got["num_tokens"][0]) == ref["num_tokens"]
    np.testing.assert_array_equal(got["status"], ref["status"])


@pytest.mark.parametrize("dtype,V,N,gamma,mask", [
    (synth.F32, 1024, 12, 7, False), (synth.BF16, 4096, 9, 5, True), (synth.F32, 8, 5, 3, False),
    (synth.F32, 40_008, 3, 2, True), (synth.BF16, 129_280, 2, 7, False)])
def test_stats_matches_oracle(ds, oracle, dtype, V, N, gamma, mask):
    w = synth.training_stats(V=V, N=N, gamma=gamma, dtype=dtype, disjoint_frac=0.1, with_mask=mask,
                             seed=V + N)
    _compare(_run(ds, w), _oracle(oracle, w))


def test_stats_special_rows(ds, oracle):
    w = synth.training_stats(V=256, N=4, gamma=3, disjoint_frac=0.0, seed=5)
    w.draft[0, 1] = w.target[0, 1]                # identical rows: L1 0, accept 1
    w.target[1, 2, 7] = float("nan")              # non-finite -> status 1
    w.labels[2, 0] = 256                          # label out of range -> status 5
    w.draft[3, 0, :] = -1e4                       # disjoint one-hot rows
    w.target[3, 0, :] = -1e4
    w.draft[3, 0, 3] = 0.0
    w.target[3, 0, 9] = 0.0
    got, ref = _run(ds, w), _oracle(oracle, w)
    assert got["status"].tolist() == ref["status"].tolist() == [0, 1, 5, 0]
    assert got["l1"][0, 1] == pytest.approx(0.0, abs=ATOL) and got["accept"][0, 1] == pytest.approx(1.0)
    assert got["l1"][3, 0] == pytest.approx(2.0, abs=ATOL) and got["accept"][3, 0] == 0.0
    ok = np.array([0, 3])
    np.testing.assert_allclose(got["l1"][ok], ref["l1"][ok], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(got["tau"][ok], ref["tau"][ok], atol=ATOL, rtol=RTOL)
    assert math.isnan(got["loss_num"][0]) and math.isnan(ref["loss_num"][0])


def test_stats_repeat_is_bitwise_identical(ds):
    w = synth.training_stats(V=8192, N=64, gamma=7, device="cuda", seed=3)
    a = ds.accept_stats(w.draft, w.target, w.labels, w.conf_logits)
    b = ds.accept_stats(w.draft, w.target, w.labels, w.conf_logits)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_stats_full_size_sampled(ds, oracle):
    """The 4096 x 7 x 129,280 fp32 workload: whole blocks sampled against the
    oracle; at every position, the disjoint rows give L1 = 2 and accept = 0;
    the numerators equal the weighted sums of the per-position outputs."""
    w = synth.training_stats(device="cuda")
    got = ds.accept_stats(w.draft, w.target, w.labels, w.conf_logits)
    torch.cuda.synchronize()
    l1, acc, tau = got["l1"].cpu().double(), got["accept"].cpu().double(), got["tau"].cpu().double()
    dis = torch.tensor(w.extra["disjoint_rows"])
    assert torch.all((l1.view(-1)[dis] - 2.0).abs() < ATOL) and torch.all(acc.view(-1)[dis] == 0.0)
    # sampled whole blocks (all gamma positions, for tau)
    blocks = sorted(set([0, w.N - 1] + torch.randint(0, w.N, (10,), generator=torch.Generator().manual_seed(1)).tolist()
                    + [int(dis[0]) // w.gamma]))
    sub = synth.StatsWorkload("sub", len(blocks), w.gamma, w.V, w.dtype, w.draft[blocks].cpu(),
                              w.target[blocks].cpu(), w.labels[blocks].cpu(), w.conf_logits[blocks].cpu(), None)
    ref = _oracle(oracle, sub)
    np.testing.assert_allclose(l1[blocks].numpy(), ref["l1"], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(acc[blocks].numpy(), ref["accept"], atol=ATOL, rtol=RTOL)
    np.testing.assert_allclose(tau[blocks].numpy(), ref["tau"], atol=ATOL, rtol=RTOL)
    # numerators vs the per-position outputs (any size)
    wk = torch.exp(-torch.arange(1, w.gamma + 1, dtype=torch.float64) / w.gamma)
    np.testing.assert_allclose(float(got["loss_num"][1]), float((l1 * wk).sum()), rtol=1e-9)
    np.testing.assert_allclose(float(got["report"][0]), float(acc.sum()), rtol=1e-9)
    np.testing.assert_allclose(float(got["report"][1]), float(tau.sum()), rtol=1e-6)
    assert int(got["num_tokens"][0]) == w.N * w.gamma
    assert int((got["status"] != 0).sum()) == 0
