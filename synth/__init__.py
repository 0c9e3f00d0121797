"""Seeded synthetic inputs shared by the tests, the smoke check and the
benchmark.

This module holds input recipes only: random logits, Zipf-shaped offsets,
planted ties and adversarial draft mass, model tables, policies and keys.  It
computes nothing the method computes (no softmax, no truncation, no sampling
rule, no acceptance), so the oracle and the CUDA library both take their
inputs from here without sharing any of the method's arithmetic.

Generation runs on a torch device: the CPU for the sizes the oracle handles,
the GPU for full-size workloads (the same recipe; the bytes depend on the
device and the torch version, so a test always hands one generated copy to
both sides).

bf16 tensors are generated as torch.bfloat16 (round to nearest even).  The
helpers ``bf16_bits`` / ``from_bf16_bits`` move them to and from the uint16 bit
patterns the oracle reads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BF16, F32 = 0, 1
VOCAB = 129_280


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A bfloat16 tensor's bit patterns as a uint16 numpy array (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bf16_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def host(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy in the oracle's layout (bf16 -> uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().contiguous().numpy()


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device, dtype=torch.float32):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def zipf_offset(rows: int, V: int, g, device, s: float = 1.1) -> torch.Tensor:
    """-s * ln(rank) with rank a per-row random permutation of 1..V (a Zipf(s)
    token-frequency profile placed at random token ids)."""
    perm = torch.argsort(torch.rand((rows, V), generator=g, device=device), dim=1)
    return -s * torch.log((perm + 1).to(torch.float32))


@dataclass
class Policy:
    temperature: torch.Tensor  # float32 [B]
    top_k: torch.Tensor        # int32 [B]
    top_p: torch.Tensor        # float32 [B]
    greedy: torch.Tensor       # int32 [B]

    def to(self, device) -> "Policy":
        return Policy(*(t.to(device) for t in (self.temperature, self.top_k, self.top_p, self.greedy)))

    def numpy(self) -> dict:
        return dict(temperature=self.temperature.cpu().numpy(), top_k=self.top_k.cpu().numpy(),
                    top_p=self.top_p.cpu().numpy(), greedy=self.greedy.cpu().numpy())

    def packed(self) -> torch.Tensor:
        """The four fields interleaved per request as 16-byte records
        (float32 temperature, int32 top_k, float32 top_p, int32 greedy)."""
        B = self.temperature.shape[0]
        rec = torch.empty((B, 4), dtype=torch.int32, device=self.temperature.device)
        rec[:, 0] = self.temperature.to(torch.float32).view(torch.int32)
        rec[:, 1] = self.top_k.to(torch.int32)
        rec[:, 2] = self.top_p.to(torch.float32).view(torch.int32)
        rec[:, 3] = self.greedy.to(torch.int32)
        return rec


def uniform_policy(B, temperature=1.0, top_k=0, top_p=1.0, greedy=False, device="cpu") -> Policy:
    return Policy(torch.full((B,), float(temperature), dtype=torch.float32, device=device),
                  torch.full((B,), int(top_k), dtype=torch.int32, device=device),
                  torch.full((B,), float(top_p), dtype=torch.float32, device=device),
                  torch.full((B,), int(bool(greedy)), dtype=torch.int32, device=device))


@dataclass
class Keys:
    seed: torch.Tensor        # uint64 as int64 [B]
    request_id: torch.Tensor  # int64 [B]
    pos0: torch.Tensor        # int64 [B]

    def numpy(self) -> dict:
        return dict(seed=self.seed.cpu().numpy().view(np.uint64),
                    request_id=self.request_id.cpu().numpy().view(np.uint64),
                    pos0=self.pos0.cpu().numpy())

    def to(self, device) -> "Keys":
        return Keys(self.seed.to(device), self.request_id.to(device), self.pos0.to(device))


def make_keys(B, seed=0, pos0=0, device="cpu", first_request=0) -> Keys:
    return Keys(torch.full((B,), int(seed), dtype=torch.int64, device=device),
                torch.arange(first_request, first_request + B, dtype=torch.int64, device=device),
                torch.full((B,), int(pos0), dtype=torch.int64, device=device))


@dataclass
class MarkovWeights:
    U: torch.Tensor | None   # bf16 [V, r]
    W: torch.Tensor | None   # bf16 [V, r]  (row v = column v of the r x V matrix)
    E: torch.Tensor | None   # bf16 [V, H]
    w_conf: torch.Tensor | None  # float32 [2H]

    @property
    def r(self) -> int:
        return 0 if self.U is None else self.U.shape[1]

    @property
    def H(self) -> int:
        return 0 if self.E is None else self.E.shape[1]


def markov_weights(V, r, H, g, device, w_std=None) -> MarkovWeights:
    U = _normal((V, r), 0.02, g, device, torch.bfloat16) if r else None
    W = _normal((V, r), 0.02, g, device, torch.bfloat16) if r else None
    if H:
        E = _normal((V, H), 0.02, g, device, torch.bfloat16)
        w = _normal((2 * H,), w_std if w_std is not None else 1.0 / math.sqrt(2 * H), g, device)
    else:
        E = w = None
    return MarkovWeights(U, W, E, w)


@dataclass
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    dtype: int
    target: torch.Tensor            # [B, gamma+1, V]
    backbone: torch.Tensor          # [B, gamma, V]
    anchor: torch.Tensor            # int32 [B]
    weights: MarkovWeights
    h: torch.Tensor | None          # [B, gamma, H]
    policy: Policy
    keys: Keys
    extra: dict = field(default_factory=dict)


def _logit_dtype(dtype):
    return torch.bfloat16 if dtype == BF16 else torch.float32


def _anchors(B, V, g, device):
    return torch.randint(0, V, (B,), generator=g, device=device, dtype=torch.int64).to(torch.int32)


# ---------------------------------------------------------------- workloads
def tiny(V=1024, B=4, gamma=5, r=16, H=64, greedy=False, device="cpu", seed=1001) -> Workload:
    """Tiny CPU-checkable case: fp32 logits, target i.i.d. N(0, 2), draft
    backbone row k = target row k-1 + N(0, 0.5); U, W, E ~ N(0, 0.02);
    h ~ N(0, 1); w ~ N(0, 1/sqrt(2H)); T = 1 with no truncation, or greedy;
    Philox seed 0, request_id = b, pos0 = 0."""
    g = _gen(seed, device)
    target = _normal((B, gamma + 1, V), 2.0, g, device)
    backbone = target[:, :gamma, :] + _normal((B, gamma, V), 0.5, g, device)
    wts = markov_weights(V, r, H, g, device)
    h = _normal((B, gamma, H), 1.0, g, device) if H else None
    return Workload("tiny", B, gamma, V, F32, target.contiguous(), backbone.contiguous(),
                    _anchors(B, V, g, device), wts, h,
                    uniform_policy(B, 1.0, 0, 1.0, greedy, device), make_keys(B, 0, 0, device))


def zipf_logits(B, rows, V, g, device, std=3.0):
    return _normal((B, rows, V), std, g, device) + zipf_offset(B * rows, V, g, device).view(B, rows, V)


def decode_verify_tile(V=VOCAB, B=64, gamma=5, r=256, H=4096, device="cpu", seed=1002,
                       sigmas=(0.3, 1.0, 3.0)) -> Workload:
    """Decode verify tile: bf16 logits; target = N(0, 3) + Zipf(1.1) per-row
    offset; draft backbone row k = target row k-1 + N(0, sigma_b) with
    sigma_b = sigmas[b mod 3]; T = 0.7, top-k 50, top-p 0.95; Markov rank r,
    draft hidden H with a random confidence weight."""
    g = _gen(seed, device)
    target = zipf_logits(B, gamma + 1, V, g, device)
    sig = torch.tensor([sigmas[b % len(sigmas)] for b in range(B)], device=device).view(B, 1, 1)
    backbone = target[:, :gamma, :] + _normal((B, gamma, V), 1.0, g, device) * sig
    wts = markov_weights(V, r, H, g, device)
    h = _normal((B, gamma, H), 1.0, g, device, torch.bfloat16) if H else None
    pos0 = torch.randint(0, 16384, (B,), generator=g, device=device, dtype=torch.int64)
    keys = Keys(torch.full((B,), 2, dtype=torch.int64, device=device),
                torch.arange(B, dtype=torch.int64, device=device), pos0)
    return Workload("decode_verify_tile", B, gamma, V, BF16,
                    target.to(torch.bfloat16).contiguous(), backbone.to(torch.bfloat16).contiguous(),
                    _anchors(B, V, g, device), wts, h,
                    uniform_policy(B, 0.7, 50, 0.95, False, device), keys)


def full_decode_tile(V=VOCAB, B=64, gamma=7, device="cpu", seed=1003, tie_frac=0.05) -> Workload:
    """Full decode tile: B requests x (1 anchor + gamma proposals) target rows,
    bf16, generated as the decode verify tile with sigma = 1; greedy only,
    no Markov head (r = 0).  In tie_frac of the target rows (chosen by seed)
    the row maximum is copied into 1-3 other random token ids; in half of
    those rows one of the copies lands on the draft row's argmax token, so
    the proposal meets an exact tie at a higher or lower index."""
    g = _gen(seed, device)
    target = zipf_logits(B, gamma + 1, V, g, device).to(torch.bfloat16)
    backbone = (target[:, :gamma, :].float() + _normal((B, gamma, V), 1.0, g, device)).to(torch.bfloat16)
    rows = B * (gamma + 1)
    n_tie = max(1, int(round(tie_frac * rows)))
    tie_rows = torch.randperm(rows, generator=g, device=device)[:n_tie].tolist()
    tflat = target.view(rows, V)
    # the draft argmax of every backbone row (the token a greedy draft proposes
    # for the next position) - used only to place planted ties
    draft_top = backbone.float().argmax(dim=2).cpu()
    n_copies = torch.randint(1, 4, (n_tie,), generator=g, device=device).tolist()
    coin = torch.rand((n_tie,), generator=g, device=device).tolist()
    spots = torch.randint(0, V, (n_tie, 3), generator=g, device=device).tolist()
    for t, row in enumerate(tie_rows):
        b, i = divmod(row, gamma + 1)
        top = tflat[row].float().max()
        idx = spots[t][: n_copies[t]]
        if coin[t] < 0.5 and i < gamma:
            idx[0] = int(draft_top[b, i])
        for v in idx:
            tflat[row, v] = top.to(torch.bfloat16)
    keys = make_keys(B, 3, 0, device)
    return Workload("full_decode_tile", B, gamma, V, BF16, target.contiguous(), backbone.contiguous(),
                    _anchors(B, V, g, device), MarkovWeights(None, None, None, None), None,
                    uniform_policy(B, 1.0, 0, 1.0, True, device), keys,
                    extra=dict(tie_rows=tie_rows))


def mixed_serving(V=VOCAB, B=256, gamma=5, r=256, H=4096, device="cpu", seed=1005,
                  adversarial_frac=0.10) -> Workload:
    """Mixed-policy serving batch: generated as the decode verify tile; per
    request T ~ U[0.3, 1.5], top-k from {0, 20, 100, 1000}, top-p from
    {1.0, 0.9, 0.8}, 25 % greedy; in adversarial_frac of the requests every
    draft backbone row puts target-max + 4 on the 8 tokens of lowest Zipf
    frequency (tokens the target's truncated policy leaves out)."""
    g = _gen(seed, device)
    ranks = torch.argsort(torch.rand((B * (gamma + 1), V), generator=g, device=device), dim=1)
    target = (_normal((B, gamma + 1, V), 3.0, g, device)
              - 1.1 * torch.log((ranks + 1).to(torch.float32)).view(B, gamma + 1, V))
    sig = torch.tensor([(0.3, 1.0, 3.0)[b % 3] for b in range(B)], device=device).view(B, 1, 1)
    backbone = target[:, :gamma, :] + _normal((B, gamma, V), 1.0, g, device) * sig
    n_adv = int(round(adversarial_frac * B))
    adv = torch.randperm(B, generator=g, device=device)[:n_adv].tolist()
    rk = ranks.view(B, gamma + 1, V)
    for b in adv:
        for k in range(gamma):
            rare = torch.topk(rk[b, k], 8).indices       # the 8 largest ranks = rarest tokens
            backbone[b, k, rare] = target[b, k].max() + 4.0
    del ranks, rk
    T = (0.3 + 1.2 * torch.rand((B,), generator=g, device=device)).to(torch.float32)
    K = torch.tensor([0, 20, 100, 1000], device=device)[
        torch.randint(0, 4, (B,), generator=g, device=device)].to(torch.int32)
    P = torch.tensor([1.0, 0.9, 0.8], device=device)[
        torch.randint(0, 3, (B,), generator=g, device=device)].to(torch.float32)
    G = (torch.rand((B,), generator=g, device=device) < 0.25).to(torch.int32)
    wts = markov_weights(V, r, H, g, device)
    h = _normal((B, gamma, H), 1.0, g, device, torch.bfloat16) if H else None
    pos0 = torch.randint(0, 16384, (B,), generator=g, device=device, dtype=torch.int64)
    keys = Keys(torch.full((B,), 5, dtype=torch.int64, device=device),
                torch.arange(B, dtype=torch.int64, device=device), pos0)
    return Workload("mixed_serving", B, gamma, V, BF16,
                    target.to(torch.bfloat16).contiguous(), backbone.to(torch.bfloat16).contiguous(),
                    _anchors(B, V, g, device), wts, h, Policy(T, K, P, G), keys,
                    extra=dict(adversarial=adv))


@dataclass
class GruWeights:
    Wi: torch.Tensor  # bf16 [3r, r], gate rows r, z, n
    Wh: torch.Tensor  # bf16 [3r, r]
    bi: torch.Tensor  # fp32 [3r]
    bh: torch.Tensor  # fp32 [3r]


def gru_weights(r, g, device, scale=None) -> GruWeights:
    """The RNN head's GRU cell at rank r: weights N(0, 1/r) (the usual
    1/sqrt(fan-in) scale), biases N(0, 0.1^2)."""
    sc = scale if scale is not None else 1.0 / r ** 0.5
    return GruWeights(_normal((3 * r, r), sc, g, device, torch.bfloat16).contiguous(),
                      _normal((3 * r, r), sc, g, device, torch.bfloat16).contiguous(),
                      _normal((3 * r,), 0.1, g, device).contiguous(),
                      _normal((3 * r,), 0.1, g, device).contiguous())


@dataclass
class StsLog:
    N: int
    gamma: int
    conf_logits: torch.Tensor  # fp32 [N, gamma]
    labels: torch.Tensor       # fp32 [N, gamma], 0 / 1 acceptances
    mask: torch.Tensor         # uint8 [N, gamma]
    temperature: torch.Tensor  # fp32 [gamma]: the miscalibration the labels were drawn with


def sts_log(N=4_194_304, gamma=7, device="cpu", seed=1008, counted=0.9) -> StsLog:
    """A serving log for Sequential Temperature Scaling: confidence logits
    N(0, 2^2) per block position, observed 0 / 1 acceptances drawn as
    Bernoulli(sigmoid(z / T_k)) with T_k spread over 0.6..3 (an over- to
    under-confident head), and a mask counting `counted` of the pairs."""
    g = _gen(seed, device)
    z = _normal((N, gamma), 2.0, g, device)
    T = torch.linspace(0.6, 3.0, gamma, device=device)
    a = (torch.rand((N, gamma), generator=g, device=device) < torch.sigmoid(z / T)).to(torch.float32)
    m = (torch.rand((N, gamma), generator=g, device=device) < counted).to(torch.uint8)
    return StsLog(N, gamma, z.contiguous(), a.contiguous(), m.contiguous(), T)


def verify_widths(B, gamma, seed=1007, invalid=0, device="cpu") -> torch.Tensor:
    """Per-request verify widths, int32 [B]: uniform over 0..gamma (a
    scheduler's choice of how many proposals to check; the pages pick it from
    measured costs, so every width is equally exercised here), with `invalid`
    requests (chosen by seed) at -1 or gamma + 1."""
    g = _gen(seed, "cpu")
    w = torch.randint(0, gamma + 1, (B,), generator=g, dtype=torch.int32)
    bad = torch.randperm(B, generator=g)[:invalid]
    w[bad] = torch.where(torch.arange(len(bad)) % 2 == 0, -1, gamma + 1).to(torch.int32)
    return w.to(device)


FLAT_POLICIES = ((1.0, 0, 0.9), (1.0, 5000, 1.0), (1.0, 5000, 0.9), (1.3, 0, 0.5),
                 (0.8, 0, 0.95), (1.0, 0, 1.0), (2.0, 300, 0.9), (1.0, 20000, 0.99))


def flat_rows(V=VOCAB, B=8, gamma=3, dtype=BF16, r=0, device="cpu", seed=1006) -> Workload:
    """Flat rows: target logits i.i.d. N(0, 0.5), so that thousands of tokens
    share a 1/8 step of (zmax - z)/T near a top-p or top-k cut (and, in bf16,
    ties hundreds deep); draft backbone row k = target row k + N(0, 0.3);
    request b takes (T, top-k, top-p) = FLAT_POLICIES[b mod 8]."""
    g = _gen(seed, device)
    target = _normal((B, gamma + 1, V), 0.5, g, device)
    backbone = target[:, :gamma, :] + _normal((B, gamma, V), 0.3, g, device)
    pol = [FLAT_POLICIES[b % len(FLAT_POLICIES)] for b in range(B)]
    policy = Policy(torch.tensor([t for t, _, _ in pol], dtype=torch.float32, device=device),
                    torch.tensor([k for _, k, _ in pol], dtype=torch.int32, device=device),
                    torch.tensor([p for _, _, p in pol], dtype=torch.float32, device=device),
                    torch.zeros((B,), dtype=torch.int32, device=device))
    td = torch.bfloat16 if dtype == BF16 else torch.float32
    return Workload("flat_rows", B, gamma, V, dtype, target.to(td).contiguous(), backbone.to(td).contiguous(),
                    _anchors(B, V, g, device), markov_weights(V, r, 0, g, device), None, policy,
                    make_keys(B, 9, 100, device))


@dataclass
class StatsWorkload:
    name: str
    N: int
    gamma: int
    V: int
    dtype: int
    draft: torch.Tensor        # [N, gamma, V]
    target: torch.Tensor       # [N, gamma, V]
    labels: torch.Tensor       # int32 [N, gamma]
    conf_logits: torch.Tensor  # float32 [N, gamma]
    mask: torch.Tensor | None  # uint8 [N, gamma]
    extra: dict = field(default_factory=dict)


def training_stats(V=VOCAB, N=4096, gamma=7, dtype=F32, device="cpu", seed=1004,
                   disjoint_frac=0.01, with_mask=False) -> StatsWorkload:
    """Training-side statistics: target t and noise e ~ N(0, 2);
    draft = rho t + sqrt(1 - rho^2) e with rho = {0, 0.5, 0.95}[n mod 3];
    disjoint_frac of the rows (by seed) are disjoint one-hot rows (0 at
    token a in the draft and b != a in the target, -1e4 elsewhere); labels are
    target-distributed draws (Gumbel-max on the target logits); confidence
    logits ~ N(0, 1); mask all ones unless with_mask (then ~10 % zeros)."""
    g = _gen(seed, device)
    rho = torch.tensor([(0.0, 0.5, 0.95)[n % 3] for n in range(N)], device=device).view(N, 1, 1)
    t = _normal((N, gamma, V), 2.0, g, device)
    d = rho * t + torch.sqrt(1.0 - rho * rho) * _normal((N, gamma, V), 2.0, g, device)
    rows = N * gamma
    n_dis = max(1, int(round(disjoint_frac * rows))) if disjoint_frac > 0 else 0
    dis = torch.randperm(rows, generator=g, device=device)[:n_dis]
    if n_dis:
        a = torch.randint(0, V, (n_dis,), generator=g, device=device)
        b = (a + torch.randint(1, V, (n_dis,), generator=g, device=device)) % V
        dv, tv = d.view(rows, V), t.view(rows, V)
        dv[dis] = -1e4
        tv[dis] = -1e4
        dv[dis, a] = 0.0
        tv[dis, b] = 0.0
    # Gumbel-max draw: argmax(t + G) with G ~ Gumbel(0, 1)
    labels = torch.empty((rows,), dtype=torch.int32, device=device)
    tv = t.view(rows, V)
    chunk = 256
    for s in range(0, rows, chunk):
        u = torch.rand((min(chunk, rows - s), V), generator=g, device=device).clamp_(min=1e-20)
        labels[s:s + chunk] = (tv[s:s + chunk] - torch.log(-torch.log(u))).argmax(dim=1).to(torch.int32)
    conf = _normal((N, gamma), 1.0, g, device)
    mask = ((torch.rand((N, gamma), generator=g, device=device) > 0.1).to(torch.uint8)
            if with_mask else None)
    ld = _logit_dtype(dtype)
    return StatsWorkload("training_stats", N, gamma, V, dtype, d.to(ld).contiguous(),
                         t.to(ld).contiguous(), labels.view(N, gamma), conf, mask,
                         extra=dict(disjoint_rows=dis.tolist()))
