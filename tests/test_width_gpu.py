"""GPU parity of the verify over a per-request width (dspark_verify_width)
against the oracle.

Greedy verify (no policy) is compared bit-exactly.  Sampled verify is compared
exactly wherever the oracle marks a request determinate, as in the fixed-width
parity tests.  Rows past a request's width hold NaN and its proposals past the
width lie outside [0, V): neither may affect it.  Width gamma must reproduce
dspark_verify, and a width call must leave the workspace ready for the next
call."""
import numpy as np
import pytest
import torch

import synth

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


def _plant_past_width(target, x, width, every=3):
    """In every `every`-th request with 0 <= w < gamma: NaN in each row past
    w, and out-of-range proposals past x_w."""
    gamma = x.shape[1]
    V = target.shape[2]
    n = 0
    for b in range(0, x.shape[0], every):
        w = int(width[b])
        if 0 <= w < gamma:
            target[b, w + 1:, 7] = float("nan")
            x[b, w:] = V + 3
            n += 1
    return n


def _host(out):
    torch.cuda.synchronize()
    return tuple(t.cpu().numpy() for t in out)


def _exact(ref, got):
    out, nacc, st = got
    np.testing.assert_array_equal(st, ref["status"])
    np.testing.assert_array_equal(nacc, ref["num_accepted"])
    np.testing.assert_array_equal(out, ref["out_tokens"])


def _determinate(ref, got, max_indet_frac):
    out, nacc, st = got
    np.testing.assert_array_equal(st, ref["status"])
    det = ~ref["indet"]
    assert det.mean() >= 1 - max_indet_frac, f"{(~det).sum()} indeterminate of {det.size}"
    np.testing.assert_array_equal(nacc[det], ref["num_accepted"][det])
    np.testing.assert_array_equal(out[det], ref["out_tokens"][det])
    # an indeterminate request: the tokens emitted before its first
    # indeterminate decision, and num_accepted when decided before it
    for b in np.flatnonzero(~det):
        n = int(ref["det_tokens"][b])
        np.testing.assert_array_equal(out[b, :n], ref["out_tokens"][b, :n], err_msg=f"request {b}")
        if ref["det_nacc"][b]:
            assert nacc[b] == ref["num_accepted"][b], b


@pytest.mark.parametrize("B,gamma,V,dtype", [
    (48, 5, 4096, torch.bfloat16), (17, 7, 40_008, torch.float32), (64, 7, 129_280, torch.bfloat16),
    (9, 1, 8, torch.float32)])
def test_width_greedy(ds, oracle, B, gamma, V, dtype):
    """Greedy prefixes over random widths 0..gamma (and two invalid ones),
    with 30 % of the proposals replaced so that prefixes end everywhere."""
    g = torch.Generator().manual_seed(B * 7 + V)
    t = (torch.randn((B, gamma + 1, V), generator=g) * 2).to(dtype)
    x = t.float().argmax(dim=2)[:, :gamma].to(torch.int32)
    flip = torch.rand((B, gamma), generator=g) < 0.3
    x[flip] = torch.randint(0, V, (int(flip.sum()),), generator=g, dtype=torch.int32)
    width = synth.verify_widths(B, gamma, seed=B + V, invalid=2)
    _plant_past_width(t, x, width)
    ref = oracle.verify(synth.host(t), x.numpy(), None, None, synth.uniform_policy(B, greedy=True).numpy(),
                        **synth.make_keys(B).numpy(), width=width.numpy())
    got = _host(ds.verify(t.cuda(), x.cuda(), width=width.cuda()))
    _exact(ref, got)
    assert (ref["status"] == 5).sum() == 2
    ok = ref["status"] == 0
    assert (ref["num_accepted"][ok] <= width.numpy()[ok]).all()


def test_width_gamma_is_dspark_verify(ds, oracle):
    """Width gamma for every request reproduces dspark_verify on the GPU, on
    the greedy path and on the sampled path."""
    w = synth.decode_verify_tile(V=4096, B=24, r=0, H=0)
    d = oracle.markov_sample(synth.host(w.backbone), w.anchor.cpu().numpy(), None, None, None, None, None,
                             w.policy.numpy(), **w.keys.numpy())
    dev = torch.device("cuda")
    t, x = w.target.to(dev), torch.from_numpy(d["proposals"]).to(dev)
    full = torch.full((w.B,), w.gamma, dtype=torch.int32).to(dev)
    _exact_pair = lambda a, b: [np.testing.assert_array_equal(u, v) for u, v in zip(a, b)]
    _exact_pair(_host(ds.verify(t, x)), _host(ds.verify(t, x, width=full)))
    kw = dict(q=torch.from_numpy(d["q"]).to(dev), q_at_x=torch.from_numpy(d["q_at_x"]).to(dev),
              policy=w.policy.packed().to(dev), seed=w.keys.seed.to(dev), request_id=w.keys.request_id.to(dev),
              pos0=w.keys.pos0.to(dev))
    _exact_pair(_host(ds.verify(t, x, **kw)), _host(ds.verify(t, x, width=full, **kw)))


@pytest.mark.parametrize("maker,kw,indet", [
    (synth.decode_verify_tile, dict(V=4096, B=24), 0.05),
    (synth.mixed_serving, dict(V=8192, B=96, adversarial_frac=0.1), 0.05),
    (synth.decode_verify_tile, dict(V=129_280, B=16), 0.10)])
def test_width_sampled(ds, oracle, maker, kw, indet):
    """Sampled verify over random widths (with two invalid ones) under the
    workload's policies; then a fixed-width call on the same workspace."""
    w = maker(r=0, H=0, **kw)
    d = oracle.markov_sample(synth.host(w.backbone), w.anchor.cpu().numpy(), None, None, None, None, None,
                             w.policy.numpy(), **w.keys.numpy())
    width = synth.verify_widths(w.B, w.gamma, seed=w.B + w.V, invalid=2)
    t = w.target.clone()
    x = torch.from_numpy(d["proposals"].copy())
    assert _plant_past_width(t, x, width) > 0
    ref = oracle.verify(synth.host(t), x.numpy(), d["q"], d["q_at_x"], w.policy.numpy(), **w.keys.numpy(),
                        width=width.numpy())
    dev = torch.device("cuda")
    args = dict(q=torch.from_numpy(d["q"]).to(dev), q_at_x=torch.from_numpy(d["q_at_x"]).to(dev),
                policy=w.policy.packed().to(dev), seed=w.keys.seed.to(dev),
                request_id=w.keys.request_id.to(dev), pos0=w.keys.pos0.to(dev))
    wsp = ds.Workspace()
    got = _host(ds.verify(t.to(dev), x.to(dev), width=width.to(dev), workspace=wsp, **args))
    _determinate(ref, got, indet)
    assert (ref["status"] == 5).sum() == 2
    # the workspace is zero-filled again: a fixed-width call on it is exact
    ref2 = oracle.verify(synth.host(w.target), d["proposals"], d["q"], d["q_at_x"], w.policy.numpy(),
                         **w.keys.numpy())
    got2 = _host(ds.verify(w.target.to(dev), torch.from_numpy(d["proposals"]).to(dev), workspace=wsp, **args))
    _determinate(ref2, got2, indet)
