"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each test checks a closed form,
a value the pages print, a library routine the case reduces to, an invariant,
a brute-force enumeration on a tiny input, or a sampling law by chi-square.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")


def _softmax64(z, T=1.0):
    inv_t = float(np.float32(1.0) / np.float32(T))
    return torch.softmax(torch.tensor(z, dtype=torch.float64) * inv_t, dim=0).numpy()


# ------------------------------------------------------------------ Philox
def test_philox_matches_independent_implementation(oracle):
    """Philox-4x32-10 against triton.language.philox run by triton's CPU
    interpreter: a second, independently written implementation of the
    generator published by Salmon et al. (SC'11)."""
    pytest.importorskip("triton")
    import subprocess
    import sys
    script = r'''
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl
@triton.jit
def k(seed_ptr, c_ptr, out_ptr, n: tl.constexpr):
    i = tl.arange(0, n)
    seed = tl.load(seed_ptr)
    c0 = tl.load(c_ptr + 4 * i + 0); c1 = tl.load(c_ptr + 4 * i + 1)
    c2 = tl.load(c_ptr + 4 * i + 2); c3 = tl.load(c_ptr + 4 * i + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3, 10)
    tl.store(out_ptr + 4 * i + 0, a); tl.store(out_ptr + 4 * i + 1, b)
    tl.store(out_ptr + 4 * i + 2, c); tl.store(out_ptr + 4 * i + 3, d)
cases = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cases:
    s = torch.tensor([seed], dtype=torch.int64)
    c = torch.tensor(ctrs, dtype=torch.int64).to(torch.int32)
    out = torch.empty(len(ctrs), dtype=torch.int32)
    k[(1,)](s, c, out, n=len(ctrs) // 4)
    res.append([x & 0xFFFFFFFF for x in out.tolist()])
print(json.dumps(res))
'''
    rng = np.random.default_rng(7)
    cases = []
    for seed in [0, 1, 0x0123456789ABCDEF, 0x7FFFFFFFFFFFFFFF, int(rng.integers(0, 2**62))]:
        ctr = rng.integers(0, 2**32, size=64 * 4, dtype=np.uint64)
        ctr[:4] = 0
        ctr[4:8] = 0xFFFFFFFF
        ctr = [int(c) - (1 << 32) if c >= (1 << 31) else int(c) for c in ctr]  # as int32
        cases.append([seed, ctr])
    env = dict(os.environ, TRITON_INTERPRET="1")
    run = subprocess.run([sys.executable, "-c", script], input=json.dumps(cases),
                         capture_output=True, text=True, env=env, timeout=600)
    assert run.returncode == 0, run.stderr[-2000:]
    expect = json.loads(run.stdout.strip().splitlines()[-1])
    for (seed, ctr), want in zip(cases, expect):
        key0, key1 = seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF
        for i in range(len(ctr) // 4):
            got = oracle.philox4x32_10(key0, key1, [c & 0xFFFFFFFF for c in ctr[4 * i: 4 * i + 4]])
            assert got.tolist() == want[4 * i: 4 * i + 4]


def test_uniform_law(oracle):
    """u = top 24 bits / 2^24: on a lattice of 2^-24, in [0, 1), uniform
    (chi-square over 1024 bins) and without lag-1 correlation."""
    n = 1 << 17
    us = np.array([oracle.uniform(12345, 6789, pos, pos % 3) for pos in range(n)])
    assert us.min() >= 0.0 and us.max() < 1.0
    assert np.all(us * 2**24 == np.floor(us * 2**24))
    from scipy import stats
    counts = np.bincount((us * 1024).astype(int), minlength=1024)
    assert stats.chisquare(counts).pvalue > 1e-4
    r = np.corrcoef(us[:-1], us[1:])[0, 1]
    assert abs(r) < 4.0 / math.sqrt(n)
    # distinct keys give distinct streams
    a = [oracle.uniform(1, 0, 5, 0), oracle.uniform(2, 0, 5, 0), oracle.uniform(1, 1, 5, 0),
         oracle.uniform(1, 0, 6, 0), oracle.uniform(1, 0, 5, 1)]
    assert len(set(a)) == 5


# ------------------------------------------------------------------ policy
@pytest.mark.parametrize("T", [1.0, 0.7, 1.5])
def test_policy_untruncated_is_library_softmax(oracle, T):
    rng = np.random.default_rng(1)
    z = rng.normal(0, 3, 500)
    st, p, am, sup, ind = oracle.policy_row(z, temperature=T)
    assert st == oracle.OK and sup == 500 and not ind
    np.testing.assert_allclose(p, _softmax64(z, T), rtol=1e-12, atol=1e-15)
    assert am == int(np.argmax(z))


def test_policy_topk_one_and_topp_zero_are_argmax(oracle):
    rng = np.random.default_rng(2)
    z = rng.normal(0, 1, 300)
    for kw in (dict(top_k=1), dict(top_p=1e-9), dict(top_p=0.0), dict(top_k=7, top_p=1e-6)):
        st, p, am, sup, _ = oracle.policy_row(z, temperature=0.9, **kw)
        assert st == oracle.OK and sup == 1
        assert p[int(np.argmax(z))] == 1.0 and p.sum() == 1.0


def test_policy_topk_V_is_noop(oracle):
    z = np.random.default_rng(3).normal(0, 2, 64)
    a = oracle.policy_row(z, temperature=0.8, top_k=64)[1]
    b = oracle.policy_row(z, temperature=0.8, top_k=0)[1]
    assert np.array_equal(a, b)


def test_policy_topk_exact_count_with_ties(oracle):
    """Exactly k tokens are kept even when the k-th value is tied; among tied
    tokens the lowest indices are kept."""
    z = np.zeros(40)
    z[[3, 9, 17, 25, 31]] = 5.0        # five tokens tied at the top
    z[[1, 2]] = 7.0
    st, p, am, sup, _ = oracle.policy_row(z, temperature=1.0, top_k=4)
    kept = set(np.nonzero(p)[0].tolist())
    assert sup == 4 and kept == {1, 2, 3, 9}
    assert am == 1
    np.testing.assert_allclose(p[1], p[2]) and np.testing.assert_allclose(p[3], p[9])
    np.testing.assert_allclose(p.sum(), 1.0, rtol=1e-15)


def test_policy_brute_force_tiny(oracle):
    """On V <= 7: the top-k set is exactly k tokens that dominate every
    dropped token (ties -> lower index kept); the top-p support has the
    minimum cardinality, over all 2^V subsets of the top-k set, of a set whose
    mass reaches p; p is proportional to exp(z/T) on it and sums to 1."""
    rng = np.random.default_rng(4)
    for trial in range(300):
        V = int(rng.integers(1, 8))
        z = np.round(rng.normal(0, 2, V), 1)      # rounding plants ties
        T = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.integers(0, V + 1))
        top_p = float(rng.choice([1.0, 0.95, 0.7, 0.4]))
        st, p, am, sup, ind = oracle.policy_row(z, temperature=T, top_k=k, top_p=top_p)
        assert st == oracle.OK
        if ind:
            continue
        use_k = 0 < k < V
        # --- top-k kept set, by pairwise dominance
        kept = list(range(V))
        if use_k:
            order = sorted(range(V), key=lambda i: (-z[i], i))
            kept = order[:k]
            for a in kept:
                for b in set(range(V)) - set(kept):
                    assert z[a] > z[b] or (z[a] == z[b] and a < b)
        support = set(np.nonzero(p)[0].tolist())
        assert support <= set(kept)
        # --- minimum cardinality by enumeration
        inv_t = float(np.float32(1.0) / np.float32(T))
        s = {i: math.exp((z[i] - z.max()) * inv_t) for i in kept}
        total = sum(s.values())
        if top_p < 1.0:
            best = None
            for size in range(1, len(kept) + 1):
                for sub in itertools.combinations(kept, size):
                    if sum(s[i] for i in sub) / total >= top_p:
                        best = size
                        break
                if best:
                    break
            assert len(support) == best
            assert sum(s[i] for i in support) / total >= top_p - 1e-12
        else:
            assert support == set(kept)
        mass = sum(s[i] for i in support)
        for i in support:
            assert abs(p[i] - s[i] / mass) < 1e-12
        assert abs(p.sum() - 1.0) < 1e-12
        assert am == min(i for i in range(V) if z[i] == z.max())


def test_policy_greedy_and_special_values(oracle):
    z = np.array([1.0, 4.0, -np.inf, 4.0, 2.0])
    st, p, am, sup, _ = oracle.policy_row(z, greedy=True)
    assert st == oracle.OK and am == 1 and p.tolist() == [0, 1, 0, 0, 0]
    st, p, *_ = oracle.policy_row(z, temperature=1.0)
    assert st == oracle.OK and p[2] == 0.0 and abs(p.sum() - 1) < 1e-15
    assert oracle.policy_row(np.array([1.0, np.nan]))[0] == oracle.NONFINITE
    assert oracle.policy_row(np.array([1.0, np.inf]))[0] == oracle.NONFINITE
    assert oracle.policy_row(np.full(4, -np.inf))[0] == oracle.EMPTY
    for bad in (dict(temperature=0.0), dict(temperature=-1.0), dict(top_k=-1),
                dict(temperature=float("nan")), dict(top_p=float("nan"))):
        assert oracle.policy_row(np.zeros(4), **bad)[0] == oracle.BAD_POLICY
    assert oracle.policy_row(np.zeros(4), temperature=0.0, greedy=True)[0] == oracle.OK


def test_policy_rounded_logits_flag_near_ties(oracle):
    z = np.array([1.0, 1.0 + 1e-7, 0.0])
    assert oracle.policy_row(z, greedy=True, exact_logits=False)[4]
    assert not oracle.policy_row(z, greedy=True, exact_logits=True)[4]


# ------------------------------------------------------------------ sampling
def test_sample_index_hand_cases(oracle):
    w = np.array([1.0, 1.0, 1.0, 1.0])
    assert oracle.sample_index(w, 0.3)[0] == 1          # 1.2 falls in (1, 2]
    assert oracle.sample_index(w, 0.0)[0] == 0
    assert oracle.sample_index(w, 0.999)[0] == 3
    assert oracle.sample_index(np.array([0.0, 0.0, 2.0, 0.0, 1.0]), 0.0)[0] == 2
    assert oracle.sample_index(np.array([0.0, 0.0, 2.0, 0.0, 1.0]), 0.7)[0] == 4
    i, margin = oracle.sample_index(np.array([1.0, 3.0]), 0.5)
    assert i == 1 and abs(margin - 0.25) < 1e-15
    assert oracle.sample_index(np.zeros(3), 0.5)[0] == -1


def test_sample_index_lattice_frequencies(oracle):
    """Over the full lattice of 24-bit uniforms restricted to a grid of 2^12
    points, each index is hit in proportion to its weight (exact counts for
    dyadic weights)."""
    w = np.array([1, 0, 3, 4, 0, 8], dtype=np.float64)      # total 16
    n = 1 << 12
    hits = np.zeros(6, int)
    for j in range(n):
        hits[oracle.sample_index(w, j / n)[0]] += 1
    assert hits.tolist() == [n * 1 // 16, 0, n * 3 // 16, n * 4 // 16, 0, n * 8 // 16]


# ------------------------------------------------------------------ Markov head
def test_markov_bias_is_library_matmul(oracle):
    """q at T = 1 without truncation is softmax(backbone + U[x_{k-1}] W) with
    the bias equal to a float64 library matmul; x_0 is the anchor and each
    later step conditions on the previous proposal."""
    w = synth.tiny(V=96, B=3, gamma=4, r=8, H=0)
    bb = w.backbone.numpy()
    U = w.weights.U.double()
    Wm = w.weights.W.double().T                       # r x V
    res = oracle.markov_sample(bb, w.anchor.numpy(), synth.host(w.weights.U), synth.host(w.weights.W),
                               None, None, None, w.policy.numpy(), **w.keys.numpy())
    assert (res["status"] == 0).all()
    for b in range(3):
        prev = int(w.anchor[b])
        for k in range(4):
            bias = torch.matmul(U[prev], Wm)
            zk = (torch.tensor(bb[b, k], dtype=torch.float64) + bias).float().double()
            want = torch.softmax(zk, 0).numpy()
            np.testing.assert_allclose(res["q"][b, k], want, rtol=1e-6, atol=1e-9)
            x = int(res["proposals"][b, k])
            assert res["q_at_x"][b, k] == res["q"][b, k, x]
            prev = x


def test_markov_zero_rank_and_one_hot_embedding(oracle):
    """r = 0: the proposal is the backbone argmax under greedy.  A one-hot U
    row e_j (scaled by s) makes the bias s * (column j of the r x V matrix),
    so a planted column maximum decides the greedy proposal."""
    V, B, gamma = 64, 2, 3
    rng = np.random.default_rng(5)
    bb = rng.normal(0, 1, (B, gamma, V)).astype(np.float32)
    pol = synth.uniform_policy(B, greedy=True).numpy()
    keys = synth.make_keys(B).numpy()
    res = oracle.markov_sample(bb, np.array([0, 1], np.int32), None, None, None, None, None, pol, **keys)
    assert np.array_equal(res["proposals"], bb.argmax(axis=2))
    assert np.all(res["q_at_x"] == 1.0)
    r = 4
    U = np.zeros((V, r), np.float32)
    U[:, 2] = 1.0                                       # every token embeds to e_2
    W = np.zeros((V, r), np.float32)
    W[41, 2] = 100.0                                    # column 2 of the matrix peaks at token 41
    Ub = synth.bf16_bits(torch.tensor(U).to(torch.bfloat16))
    Wb = synth.bf16_bits(torch.tensor(W).to(torch.bfloat16))
    res = oracle.markov_sample(np.zeros((B, gamma, V), np.float32), np.array([5, 7], np.int32),
                               Ub, Wb, None, None, None, pol, **keys)
    assert np.all(res["proposals"] == 41)


def test_confidence_closed_forms(oracle):
    V, B, gamma, H = 16, 2, 2, 2
    bb = np.zeros((B, gamma, V), np.float32)
    pol = synth.uniform_policy(B, greedy=True).numpy()
    keys = synth.make_keys(B).numpy()
    h = np.array([[[1.0, 2.0], [0.5, -1.0]], [[3.0, 0.0], [0.0, 0.0]]], np.float32)
    E = np.zeros((V, H), np.float32)
    E[3] = [0.25, -0.5]
    Eb = synth.bf16_bits(torch.tensor(E).to(torch.bfloat16))
    res = oracle.markov_sample(bb, np.array([3, 3], np.int32), None, None, h, Eb,
                               np.zeros(2 * H, np.float32), pol, **keys)
    assert np.all(res["conf"] == 0.5)                   # w = 0 -> sigmoid(0)
    wv = np.array([0.5, -1.0, 2.0, 4.0], np.float32)
    res = oracle.markov_sample(bb, np.array([3, 3], np.int32), None, None, h, Eb, wv, pol, **keys)
    # request 0, k = 1 conditions on the anchor 3: a = 0.5*1 - 1*2 + 2*0.25 + 4*(-0.5) = -3
    assert abs(res["conf"][0, 0] - 1 / (1 + math.exp(3.0))) < 1e-7
    # k = 2 conditions on x_1 = argmax of a zero row = token 0 (E[0] = 0): a = 0.25 + 1 = 1.25
    assert res["proposals"][0, 0] == 0
    assert abs(res["conf"][0, 1] - 1 / (1 + math.exp(-1.25))) < 1e-7


def test_markov_proposals_follow_q(oracle):
    """x_1 drawn with Philox draw 0 follows q_1 (chi-square over requests)."""
    V, B = 6, 60000
    bb = np.tile(np.array([0.0, 1.0, -1.0, 2.0, 0.5, -3.0], np.float32), (B, 1, 1))
    pol = synth.uniform_policy(B, temperature=1.0).numpy()
    keys = synth.make_keys(B, seed=99, pos0=17).numpy()
    res = oracle.markov_sample(bb, np.zeros(B, np.int32), None, None, None, None, None, pol, **keys)
    counts = np.bincount(res["proposals"][:, 0], minlength=V)
    from scipy import stats
    want = _softmax64(bb[0, 0]) * B
    assert stats.chisquare(counts, want).pvalue > 1e-3


def test_markov_bad_anchor_and_nonfinite(oracle):
    V, B, gamma = 8, 3, 2
    bb = np.zeros((B, gamma, V), np.float32)
    bb[2, 1, 3] = np.nan
    pol = synth.uniform_policy(B, greedy=True).numpy()
    res = oracle.markov_sample(bb, np.array([0, 8, 0], np.int32), None, None, None, None, None,
                               pol, **synth.make_keys(B).numpy())
    assert res["status"].tolist() == [0, oracle.BAD_TOKEN, oracle.NONFINITE]
    assert res["proposals"][1].tolist() == [-1, -1]
    assert res["proposals"][2, 1] == -1 and res["proposals"][2, 0] == 0


# ------------------------------------------------------------------ verify
def _verify_greedy_case(oracle, argmaxes, proposals, V=10):
    rows = len(argmaxes)
    t = np.zeros((1, rows, V), np.float32)
    for i, a in enumerate(argmaxes):
        t[0, i, a] = 1.0
    pol = synth.uniform_policy(1, greedy=True).numpy()
    return oracle.verify(t, np.array([proposals], np.int32), None, None, pol,
                         **synth.make_keys(1).numpy())


def test_golden_greedy_no_later_match(oracle):
    g = json.load(open(GOLDEN))["greedy_no_later_match"]
    res = _verify_greedy_case(oracle, g["target_argmax_per_row"], g["proposals"])
    n = int(res["num_accepted"][0])
    assert n == g["expected_num_accepted"]
    assert res["out_tokens"][0, : n + 1].tolist() == g["expected_emitted"]
    assert np.all(res["out_tokens"][0, n + 1:] == -1)


def test_greedy_identical_accepts_all_with_bonus(oracle):
    res = _verify_greedy_case(oracle, [4, 1, 1, 9, 0, 2], [4, 1, 1, 9, 0])
    assert res["num_accepted"][0] == 5 and res["out_tokens"][0].tolist() == [4, 1, 1, 9, 0, 2]


def test_golden_emitted_range(oracle):
    """1..gamma+1 tokens for gamma = 7, over random greedy rows."""
    g = json.load(open(GOLDEN))["emitted_range"]
    gamma, V, B = g["gamma"], 5, 4000
    rng = np.random.default_rng(8)
    t = rng.normal(0, 1, (B, gamma + 1, V)).astype(np.float32)
    a = t.argmax(axis=2)
    x = np.where(rng.random((B, gamma)) < 0.8, a[:, :gamma], rng.integers(0, V, (B, gamma))).astype(np.int32)
    res = oracle.verify(t, x, None, None, synth.uniform_policy(B, greedy=True).numpy(),
                        **synth.make_keys(B).numpy())
    emitted = res["num_accepted"] + 1
    assert emitted.min() == g["min_emitted"] and emitted.max() == g["max_emitted"]
    for b in range(B):
        n = res["num_accepted"][b]
        assert np.array_equal(x[b, :n], a[b, :n]) and (n == gamma or x[b, n] != a[b, n])
        assert res["out_tokens"][b, n] == a[b, n]


def test_greedy_ties_lowest_index(oracle):
    V = 12
    t = np.zeros((2, 2, V), np.float32)
    t[:, 0, [4, 9]] = 3.0                   # exact tie between tokens 4 and 9
    t[:, 1, 2] = 1.0
    x = np.array([[9], [4]], np.int32)      # request 0 proposes the higher tied index
    res = oracle.verify(t, x, None, None, synth.uniform_policy(2, greedy=True).numpy(),
                        **synth.make_keys(2).numpy())
    assert res["num_accepted"].tolist() == [0, 1]
    assert res["out_tokens"].tolist() == [[4, -1], [4, 2]]


def test_verify_p_equals_q_accepts_all(oracle):
    """p == q gives ratio 1 > u for every u in [0, 1): every proposal is
    accepted and the bonus comes from row gamma's support."""
    V, gamma, B = 32, 4, 500
    rng = np.random.default_rng(9)
    t = rng.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
    q = np.stack([[_softmax64(t[b, k]) for k in range(gamma)] for b in range(B)]).astype(np.float32)
    x = np.array([[rng.choice(V, p=q[b, k] / q[b, k].sum()) for k in range(gamma)] for b in range(B)], np.int32)
    qx = np.take_along_axis(q, x[..., None], 2)[..., 0]
    pol = synth.uniform_policy(B, temperature=1.0).numpy()
    # the accept ratio is p/q with p from the oracle's float64 policy and q its
    # fp32 rounding: ratio = 1 +- 1e-7, above every 24-bit uniform
    res = oracle.verify(t, x, q, qx, pol, **synth.make_keys(B, seed=3).numpy())
    assert np.all(res["num_accepted"] == gamma)
    assert np.array_equal(res["out_tokens"][:, :gamma], x)


def test_verify_disjoint_rejects_first_and_resamples_p(oracle):
    V, gamma, B = 16, 3, 400
    t = np.full((B, gamma + 1, V), -np.inf, np.float32)
    t[:, :, :8] = np.random.default_rng(10).normal(0, 1, (B, gamma + 1, 8))
    q = np.zeros((B, gamma, V), np.float32)
    q[:, :, 8:] = 1.0 / 8
    x = np.full((B, gamma), 12, np.int32)
    qx = np.full((B, gamma), 1.0 / 8, np.float32)
    res = oracle.verify(t, x, q, qx, synth.uniform_policy(B).numpy(), **synth.make_keys(B).numpy())
    assert np.all(res["num_accepted"] == 0)
    assert np.all(res["out_tokens"][:, 0] < 8)
    assert np.all(res["out_tokens"][:, 1:] == -1)


def _chi2_regime(oracle, regime, policy, seed):
    V, gamma, B = 8, 3, 200_000
    rng = np.random.default_rng(seed)
    t_logits = rng.normal(0, 1.5, (gamma + 1, V))
    if regime == "agreeing":
        d_logits = t_logits[:gamma] + rng.normal(0, 0.3, (gamma, V))
    elif regime == "disagreeing":
        d_logits = rng.normal(0, 1.5, (gamma, V))
    else:  # nearly disjoint: the target lives on 0..3, the draft mostly on 4..7
        t_logits[:, 4:] = -np.inf
        d_logits = np.full((gamma, V), 0.0)
        d_logits[:, :4] = -6.0
    t = np.tile(t_logits.astype(np.float32), (B, 1, 1))
    q_rows = np.stack([_softmax64(d_logits[k]) for k in range(gamma)])
    q = np.tile(q_rows.astype(np.float32), (B, 1, 1))
    x = np.stack([rng.choice(V, size=B, p=q_rows[k] / q_rows[k].sum()) for k in range(gamma)], 1).astype(np.int32)
    qx = np.take_along_axis(q, x[..., None], 2)[..., 0]
    pol = {k: np.full(B, v, dtype=np.float32 if k in ("temperature", "top_p") else np.int32)
           for k, v in policy.items()}
    res = oracle.verify(t, x, q, qx, pol, **synth.make_keys(B, seed=seed).numpy())
    # target-only laws: the policy applied to each target row (pinned above)
    p_rows = [oracle.policy_row(t_logits[i], **policy)[1] for i in range(2)]
    return res, p_rows


@pytest.mark.parametrize("regime", ["agreeing", "disagreeing", "nearly_disjoint"])
@pytest.mark.parametrize("policy", [dict(temperature=1.0, top_k=0, top_p=1.0),
                                    dict(temperature=0.7, top_k=6, top_p=0.9)])
def test_verify_preserves_target_law(oracle, regime, policy):
    """Emitted tokens are distributed as target-only sampling: the first
    emitted token ~ p_0, and given x_1 accepted the second ~ p_1
    (chi-square, alpha = 1e-3)."""
    import zlib
    from scipy import stats
    seed = zlib.crc32(f"{regime}-{policy['top_k']}".encode()) % 1000
    res, (p0, p1) = _chi2_regime(oracle, regime, dict(policy, greedy=0), seed=seed)
    assert np.all(res["status"] == 0)

    def law(tokens, p):
        sup = p > 0
        assert np.all(sup[tokens])                 # never outside the target support
        if sup.sum() == 1:                          # one-token support: exact
            assert np.all(tokens == np.argmax(p))
            return
        c = np.bincount(tokens, minlength=len(p))[sup]
        assert stats.chisquare(c, p[sup] * c.sum()).pvalue > 1e-3

    law(res["out_tokens"][:, 0], p0)
    sel = res["num_accepted"] >= 1
    if sel.sum() > 2000:
        law(res["out_tokens"][sel, 1], p1)


def test_verify_bonus_from_last_row(oracle):
    """With every proposal accepted, the extra token is drawn from row gamma
    (a one-hot target row there forces it)."""
    V, gamma, B = 8, 2, 50
    t = np.zeros((B, gamma + 1, V), np.float32)
    t[:, gamma, :] = -np.inf
    t[:, gamma, 6] = 0.0
    q = np.full((B, gamma, V), 1.0 / V, np.float32)
    x = np.full((B, gamma), 2, np.int32)
    res = oracle.verify(t, x, q, q[:, :, 0], synth.uniform_policy(B).numpy(), **synth.make_keys(B).numpy())
    assert np.all(res["num_accepted"] == gamma) and np.all(res["out_tokens"][:, gamma] == 6)


def test_verify_bad_inputs(oracle):
    V, gamma = 8, 2
    t = np.zeros((3, gamma + 1, V), np.float32)
    t[2, 2, 0] = np.inf
    x = np.array([[0, 9], [1, 1], [0, 0]], np.int32)
    res = oracle.verify(t, x, None, None, synth.uniform_policy(3, greedy=True).numpy(),
                        **synth.make_keys(3).numpy())
    assert res["status"].tolist() == [oracle.BAD_TOKEN, 0, oracle.NONFINITE]
    assert res["num_accepted"][0] == -1 and np.all(res["out_tokens"][0] == -1)


# ------------------------------------------------------------------ stats
def _stats(oracle, d, t, labels=None, conf=None, mask=None):
    d = np.asarray(d, np.float32)
    t = np.asarray(t, np.float32)
    N, gamma, V = d.shape
    labels = np.zeros((N, gamma), np.int32) if labels is None else labels
    conf = np.zeros((N, gamma), np.float32) if conf is None else conf
    return oracle.accept_stats(d, t, labels, conf, mask)


def test_golden_disjoint_l1_two_accept_zero(oracle):
    g = json.load(open(GOLDEN))["disjoint_l1_accept"]
    res = _stats(oracle, [g["draft_logits"]], [g["target_logits"]])
    assert res["l1"][0, 0] == g["expected_l1"]
    assert res["accept"][0, 0] == g["expected_accept_rate"]
    assert res["tau"][0] == 1.0


def test_golden_identical_tau(oracle):
    g = json.load(open(GOLDEN))["identical_tau"]
    gamma = g["gamma"]
    z = np.random.default_rng(11).normal(0, 2, (3, gamma, 50))
    res = _stats(oracle, z, z)
    assert np.all(res["l1"] == 0.0)
    assert np.all(res["accept"] == g["expected_accept_rate"])
    assert np.all(res["tau"] == g["expected_tau"])


def test_stats_two_point_closed_forms(oracle):
    """Two-point rows: L1 = 2|a - b|, accept = 1 - |a - b|; with accept 1/2
    at every position tau = 1 + sum_k 2^-k."""
    gamma = 4
    a = np.array([0.9, 0.5, 0.25, 0.8])
    b = np.array([0.4, 0.5, 0.75, 0.3])
    d = np.full((1, gamma, 6), -np.inf)
    t = np.full((1, gamma, 6), -np.inf)
    d[0, :, 1], d[0, :, 4] = np.log(a), np.log(1 - a)
    t[0, :, 1], t[0, :, 4] = np.log(b), np.log(1 - b)
    res = _stats(oracle, d, t, labels=np.full((1, gamma), 1, np.int32))
    np.testing.assert_allclose(res["l1"][0], 2 * np.abs(a - b), atol=1e-6)
    np.testing.assert_allclose(res["accept"][0], 1 - np.abs(a - b), atol=1e-6)
    acc = 1 - np.abs(a - b)
    np.testing.assert_allclose(res["tau"][0], 1 + np.cumprod(acc).sum(), rtol=1e-6)
    # CE at label 1 is -log a' where a' is a after the logits' fp32 rounding
    la, lb = np.log(a).astype(np.float32).astype(np.float64), np.log(1 - a).astype(np.float32).astype(np.float64)
    a_r = np.exp(la) / (np.exp(la) + np.exp(lb))
    w = np.exp(-np.arange(1, gamma + 1) / gamma)
    np.testing.assert_allclose(res["loss_num"][0], np.sum(w * -np.log(a_r)), rtol=1e-12)


def test_stats_ce_onehot_zero_and_uniform_logV(oracle):
    gamma, V = 3, 40
    d = np.full((2, gamma, V), -1e4)
    d[:, :, 7] = 0.0
    t = np.zeros((2, gamma, V))
    labels = np.full((2, gamma), 7, np.int32)
    res = _stats(oracle, d, t, labels=labels)
    assert res["loss_num"][0] == 0.0                       # one-hot draft at the label
    res = _stats(oracle, t, t, labels=labels)              # uniform draft: CE = log V
    w = np.exp(-np.arange(1, gamma + 1) / gamma)
    np.testing.assert_allclose(res["loss_num"][0], 2 * np.log(V) * w.sum(), rtol=1e-12)
    # the weights sum to a geometric series
    np.testing.assert_allclose(w.sum(), math.exp(-1 / gamma) * (1 - math.exp(-1)) / (1 - math.exp(-1 / gamma)))


def test_stats_bce_closed_forms(oracle):
    gamma = 2
    zc = np.array([[1.5, -2.0]], np.float32)
    d0 = np.array([[[0.0, -1e4], [0.0, -1e4]]])
    # identical rows: accept = 1 -> BCE = softplus(z) - z = softplus(-z)
    res = _stats(oracle, d0, d0, conf=zc)
    w = np.exp(-np.arange(1, gamma + 1) / gamma)
    want = np.sum(w * np.log1p(np.exp(-zc[0].astype(np.float64))))
    np.testing.assert_allclose(res["loss_num"][2], want, rtol=1e-12)
    # disjoint rows: accept = 0 -> BCE = softplus(z)
    d1 = np.array([[[-1e4, 0.0], [-1e4, 0.0]]])
    res = _stats(oracle, d0, d1, conf=zc)
    want = np.sum(w * np.log1p(np.exp(zc[0].astype(np.float64))))
    np.testing.assert_allclose(res["loss_num"][2], want, rtol=1e-12)
    np.testing.assert_allclose(res["loss_num"][3],
                               0.1 * res["loss_num"][0] + 0.9 * res["loss_num"][1] + res["loss_num"][2])


def test_stats_library_routines_and_mask(oracle):
    """Random rows: L1 from float64 library softmaxes, CE from the library
    cross-entropy, BCE from the library BCE-with-logits; the mask removes
    positions from the numerators and the token count only."""
    import torch.nn.functional as F
    N, gamma, V = 5, 3, 300
    rng = np.random.default_rng(12)
    d = rng.normal(0, 2, (N, gamma, V)).astype(np.float32)
    t = rng.normal(0, 2, (N, gamma, V)).astype(np.float32)
    y = rng.integers(0, V, (N, gamma)).astype(np.int32)
    zc = rng.normal(0, 1, (N, gamma)).astype(np.float32)
    m = (rng.random((N, gamma)) > 0.3).astype(np.uint8)
    res = oracle.accept_stats(d, t, y, zc, m)
    D, Tt = torch.tensor(d, dtype=torch.float64), torch.tensor(t, dtype=torch.float64)
    l1 = (torch.softmax(D, -1) - torch.softmax(Tt, -1)).abs().sum(-1)
    np.testing.assert_allclose(res["l1"], l1.numpy(), rtol=1e-6)
    acc = (1 - 0.5 * l1).clamp(0, 1)
    ce = F.cross_entropy(D.reshape(-1, V), torch.tensor(y, dtype=torch.long).reshape(-1),
                         reduction="none").reshape(N, gamma)
    bce = F.binary_cross_entropy_with_logits(torch.tensor(zc, dtype=torch.float64), acc, reduction="none")
    w = torch.exp(-torch.arange(1, gamma + 1, dtype=torch.float64) / gamma)
    M = torch.tensor(m, dtype=torch.float64)
    np.testing.assert_allclose(res["loss_num"][0], float((w * M * ce).sum()), rtol=1e-10)
    np.testing.assert_allclose(res["loss_num"][1], float((w * M * l1).sum()), rtol=1e-10)
    np.testing.assert_allclose(res["loss_num"][2], float((w * M * bce).sum()), rtol=1e-10)
    assert res["num_tokens"] == int(m.sum())
    np.testing.assert_allclose(res["report"][0], float((M * acc).sum()), rtol=1e-10)
    tau = 1 + torch.cumprod(acc, 1).sum(1)
    np.testing.assert_allclose(res["tau"], tau.numpy(), rtol=1e-6)
    np.testing.assert_allclose(res["report"][1], float(tau.sum()), rtol=1e-10)


def test_stats_bad_label_and_nonfinite(oracle):
    d = np.zeros((2, 1, 4), np.float32)
    t = np.zeros((2, 1, 4), np.float32)
    t[1, 0, 2] = np.nan
    res = oracle.accept_stats(d, t, np.array([[4], [0]], np.int32), np.zeros((2, 1), np.float32))
    assert res["status"].tolist() == [oracle.BAD_TOKEN, oracle.NONFINITE]
    assert math.isnan(res["loss_num"][0])


def test_synthetic_bf16_roundtrip():
    x = torch.randn(1000).to(torch.bfloat16)
    assert torch.equal(synth.from_bf16_bits(synth.bf16_bits(x)), x)
