#!/usr/bin/env python
"""Benchmark of the DSpark draft-sampling / exact-verify hot path on GB300.

One step = the whole path over one batch of synthetic input, inputs resident
in HBM when the timed region starts.  Workloads (``--workload``):

  full_decode_tile   (default; the headline metric's workload) 64 requests x
                     (1 anchor + gamma = 7) = 512 target rows, V = 129,280,
                     bf16, greedy, no Markov bias: the draft proposals (argmax
                     of the 448 draft rows) then the exact greedy verify.
  decode_verify_tile 64 requests, gamma = 5, bf16, T = 0.7 / top-k 50 /
                     top-p 0.95, Markov rank 256, draft hidden 4096: Markov
                     sampling (bias GEMM + policy + draw per position,
                     confidences) then the sampled verify.
  mixed_serving      256 requests, gamma = 5, per-request policies, 25 %
                     greedy, 10 % adversarial drafts, rank 256.
  decode_verify_tile_width  the decode verify tile with a per-request verify
                     width uniform over 0..gamma (seeded): the draft of gamma
                     positions, then the verify of x_1..x_w and the bonus from
                     row w; positions = the sum of (w + 1).
  rnn_decode_tile    the decode verify tile drafted by the RNN head instead
                     of the Markov head (a GRU state at rank 256 carried
                     across the block gives the bias), then the sampled verify.
  sts_fit            Sequential Temperature Scaling of a serving log:
                     4,194,304 blocks x gamma = 7 (confidence logit, 0 / 1
                     acceptance, mask) pairs; one whole fit per step.
  training_stats     4096 blocks x gamma = 7 fp32 row pairs: L1, accept rate,
                     tau and the weighted loss numerators.
  training_stats_grad  the same row pairs: the gradient of the loss numerators'
                     total with respect to the draft and confidence logits
                     (gradient rows written in full).

The step's inputs exceed L2 (135.5 MB on GB300) in every workload; in addition
a 2 x L2-sized read of another buffer before every timed step, outside the
step's events, evicts them (a read, so no dirty lines are left to be written
back inside the step).  Prints one JSON line.  ``--impl reference`` times the
CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import atexit
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("verified positions/s and achieved HBM GB/s (% of GB300 roofline) at "
          "512×(γ+1)×129,280")
UNIT = "positions/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_step_ms(ms, world, device):
    """The job's step time over independent replicas: the slowest rank's.
    Every rank gets the same value (no data moves between replicas)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(positions, ms, world):
    """Whole-job positions per second: every replica processes `positions`
    per step, the job's step takes `ms` (the slowest rank's)."""
    return positions * world / (ms * 1e-3)


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, path: str | None = None):
        self.dev = device_index
        self.proc = None
        # the raw samples: a temporary file unless --clocks-csv names one to keep
        self.path = path or os.path.join(tempfile.gettempdir(), f"dspark_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            atexit.register(self.__exit__, None, None, None)  # the sampler never outlives the bench
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.proc is not None and not self.f.closed:
            self.f.close()

    def summary(self, t_start=None, t_end=None):
        """Median SM clock and throttle reasons of the samples taken between
        t_start and t_end (time.time() seconds)."""
        import datetime
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                mhz, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            if t_start is not None and not (t_start <= ts <= t_end):
                continue
            sm.append(mhz)
            smax.append(mx)
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ workloads
class Serving:
    """Draft sampling then exact verify of one batch."""

    def __init__(self, name, w, esize, width=None, gru=None):
        self.name, self.w, self.esize = name, w, esize
        self.width = width  # int32 [B] verify widths, or None (gamma for every request)
        self.gru = gru      # GRU weights: the RNN head drafts instead of the Markov head
        self.positions = w.B * (w.gamma + 1) if width is None else int((width.cpu().long() + 1).sum())
        self.greedy_only = bool(w.policy.greedy.all()) and w.weights.r == 0

    def config(self):
        w = self.w
        return {"workload": self.name, "requests": w.B, "gamma": w.gamma, "vocab": w.V,
                "target_rows": w.B * (w.gamma + 1), "draft_rows": w.B * w.gamma,
                "policy": "greedy" if self.greedy_only else "per-request temperature / top-k / top-p",
                "markov_rank": w.weights.r, "draft_hidden": w.weights.H,
                **({} if self.gru is None else {"sequential_head": f"RNN (GRU, rank {w.weights.r})"}),
                **({} if self.width is None else {
                    "verify_width": f"per request, uniform over 0..{w.gamma} (seeded; mean "
                                    f"{float(self.width.float().mean()):.2f} proposals checked)",
                    "verified_rows": self.positions})}

    def setup(self, ds, dev):
        w = self.w
        B, g, V = w.B, w.gamma, w.V
        self.ds = ds
        self.ws = ds.Workspace()
        self.pol = None if self.greedy_only else w.policy.packed().to(dev)
        self.keys = dict(seed=w.keys.seed.to(dev), request_id=w.keys.request_id.to(dev), pos0=w.keys.pos0.to(dev))
        self.wts = dict(U=w.weights.U, W=w.weights.W, E=w.weights.E, w_conf=w.weights.w_conf)
        if self.gru is not None:
            self.gru_dev = dict(Wi=self.gru.Wi.to(dev), Wh=self.gru.Wh.to(dev), bi=self.gru.bi.to(dev),
                                bh=self.gru.bh.to(dev))
        self.draft_out = dict(proposals=torch.empty((B, g), dtype=torch.int32, device=dev),
                              q=None if self.pol is None else torch.empty((B, g, V), dtype=torch.float32, device=dev),
                              q_at_x=torch.empty((B, g), dtype=torch.float32, device=dev),
                              conf=torch.empty((B, g), dtype=torch.float32, device=dev) if w.h is not None else None,
                              status=torch.empty((B,), dtype=torch.int32, device=dev))
        self.ver_out = (torch.empty((B, g + 1), dtype=torch.int32, device=dev),
                        torch.empty((B,), dtype=torch.int32, device=dev),
                        torch.empty((B,), dtype=torch.int32, device=dev))
        self.width_dev = None if self.width is None else self.width.to(dev)
        # the step's inputs, in the order e2e_compute unpacks them
        self.inputs = [w.backbone, w.target, w.anchor]
        self.h_at = self.width_at = None
        if w.h is not None:
            self.h_at = len(self.inputs)
            self.inputs.append(w.h)
        if self.width_dev is not None:
            self.width_at = len(self.inputs)
            self.inputs.append(self.width_dev)

    def draft(self, stream, backbone=None, anchor=None, h=None):
        w = self.w
        d = self.draft_out
        bb = backbone if backbone is not None else w.backbone
        an = anchor if anchor is not None else w.anchor
        hh = h if h is not None else w.h
        keys = self.keys if self.pol is not None else {}
        if self.gru is not None:
            self.ds.rnn_sample(bb, an, self.wts["U"], self.wts["W"], **self.gru_dev, h=hh, E=self.wts["E"],
                               w_conf=self.wts["w_conf"], policy=self.pol, workspace=self.ws, out=d, stream=stream,
                               **keys)
        else:
            self.ds.markov_sample(bb, an, h=hh, policy=self.pol, workspace=self.ws, out=d, stream=stream,
                                  **self.wts, **keys)

    def verify(self, stream, target=None, width=None):
        d = self.draft_out
        self.ds.verify(target if target is not None else self.w.target, d["proposals"], q=d["q"],
                       q_at_x=d["q_at_x"] if self.pol is not None else None, policy=self.pol,
                       workspace=self.ws, out=self.ver_out, stream=stream,
                       width=width if width is not None else self.width_dev,
                       **(self.keys if self.pol is not None else {}))

    def parts(self):
        return [("draft", self.draft), ("verify", self.verify)]

    def bytes(self):
        """Bytes the method must move once, per part."""
        w, e = self.w, self.esize
        B, g, V, r, H = w.B, w.gamma, w.V, w.weights.r, w.weights.H
        sampled = int((self.w.policy.greedy == 0).sum()) if self.pol is not None else 0
        # the method reads the rank-r matrix once a step (the RNN head's two
        # products, hi and lo, and the z between them are this library's cost)
        draft = (B * g * V * e                      # backbone rows
                 + g * (V * r * 2 + B * r * 2)      # the rank-r matrix, gathered rows / states
                 + (0 if self.gru is None else g * 2 * 3 * r * r * 2)  # GRU weights
                 + sampled * g * V * 4              # q rows of sampled requests
                 + B * g * (H * 2 * 2 if w.h is not None else 0)  # h and E rows for c_k
                 + B * 4 + B * g * 12)              # anchors, proposals, q(x), c_k
        rejecting = 0
        checked = g if self.width is None else self.width.cpu()
        if self.pol is not None:
            nacc = self.ver_out[1].cpu()
            greedy = self.w.policy.greedy.cpu() != 0
            rejecting = int(((nacc < checked) & (nacc >= 0) & ~greedy).sum())
        # target rows 0..w of every request, the residual's q row at a
        # rejection, proposals and q(x), outputs, keys (and the widths)
        rows = self.positions
        verify = (rows * V * e + rejecting * V * 4 + B * g * 8 + B * (g + 1) * 4 + B * 8
                  + (0 if self.width is None else B * 4))
        return {"draft": draft, "verify": verify}

    def flops(self):
        w = self.w
        passes = 1 if self.gru is None else 2
        return {"draft": passes * 2 * w.B * w.weights.r * w.V * w.gamma}

    def e2e_compute(self, stream, dev_inputs, host_outputs):
        """One step through the public API on inputs just copied to the
        device, then the results read back to the host."""
        backbone, target, anchor = dev_inputs[:3]
        h = dev_inputs[self.h_at] if self.h_at is not None else None
        width = dev_inputs[self.width_at] if self.width_at is not None else None
        self.draft(stream, backbone=backbone, anchor=anchor, h=h)
        self.verify(stream, target=target, width=width)
        for h, d in zip(host_outputs, self.ver_out):
            h.copy_(d, non_blocking=True)

    def outputs(self):
        return list(self.ver_out)

    def check(self):
        st = self.ver_out[2]
        assert int((st != 0).sum()) == 0, "unexpected request failures in the benchmark workload"

    def cpu_sample(self, budget_s, max_requests=None):
        """The oracle on whole requests of the workload (draft + verify), one
        request at a time, single-threaded."""
        import oracle
        oracle.build()
        w = self.w
        bb, tg = synth.host(w.backbone), synth.host(w.target)
        anchor = w.anchor.cpu().numpy()
        keys = w.keys.numpy()
        pol = (synth.uniform_policy(w.B, greedy=True) if self.greedy_only else w.policy).numpy()
        U = synth.host(w.weights.U) if w.weights.r else None
        Wm = synth.host(w.weights.W) if w.weights.r else None
        hh = synth.host(w.h) if w.h is not None else None
        E = synth.host(w.weights.E) if w.h is not None else None
        wc = w.weights.w_conf.cpu().numpy() if w.h is not None else None
        wd = None if self.width is None else self.width.cpu().numpy().astype(np.int32)
        done, pos, b, t0 = 0, 0, 0, time.perf_counter()
        while True:
            sl = slice(b, b + 1)
            k = {n: v[sl] for n, v in keys.items()}
            p = {n: v[sl] for n, v in pol.items()}
            if self.gru is not None:
                gw = self.gru
                d = oracle.rnn_sample(bb[sl], anchor[sl], U, Wm, synth.host(gw.Wi), synth.host(gw.Wh),
                                      gw.bi.cpu().numpy(), gw.bh.cpu().numpy(), None if hh is None else hh[sl], E,
                                      wc, p, **k)
            else:
                d = oracle.markov_sample(bb[sl], anchor[sl], U, Wm, None if hh is None else hh[sl], E, wc, p, **k)
            oracle.verify(tg[sl], d["proposals"], d["q"], d["q_at_x"], p, **k,
                          width=None if wd is None else wd[sl])
            done += 1
            pos += w.gamma + 1 if wd is None else int(wd[b]) + 1
            b = (b + 1) % w.B
            el = time.perf_counter() - t0
            if el >= budget_s or (max_requests and done >= max_requests):
                break
        rows = f"{w.gamma + 1} rows each" if wd is None else "w + 1 rows each at the request's width w"
        return {"value": pos / el, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{done} whole requests of the workload (draft of {w.gamma} rows + verify of "
                          f"{rows}; {pos} verified positions) in {el:.1f} s, "
                          f"single-threaded C++ oracle"}


class Stats:
    """Acceptance statistics of one batch of row pairs."""

    def __init__(self, w, blocks=None):
        self.w = w
        self.name = "training_stats"
        self.positions = w.N * w.gamma
        self.blocks = blocks or w.N  # blocks of the workload (the CPU arm generates a subset)

    def config(self):
        w = self.w
        return {"workload": self.name, "blocks": self.blocks, "gamma": w.gamma, "vocab": w.V,
                "row_pairs": self.blocks * w.gamma, "dtype": "fp32"}

    def setup(self, ds, dev):
        w = self.w
        self.ds = ds
        self.ws = ds.Workspace()
        N, g = w.N, w.gamma
        self.out = dict(l1=torch.empty((N, g), dtype=torch.float32, device=dev),
                        accept=torch.empty((N, g), dtype=torch.float32, device=dev),
                        tau=torch.empty((N,), dtype=torch.float32, device=dev),
                        loss_num=torch.empty((4,), dtype=torch.float64, device=dev),
                        report=torch.empty((2,), dtype=torch.float64, device=dev),
                        num_tokens=torch.empty((1,), dtype=torch.int64, device=dev),
                        status=torch.empty((N,), dtype=torch.int32, device=dev))
        self.inputs = [w.draft, w.target, w.labels, w.conf_logits]

    def stats(self, stream, draft=None, target=None, labels=None, conf=None):
        w = self.w
        self.ds.accept_stats(draft if draft is not None else w.draft, target if target is not None else w.target,
                             labels if labels is not None else w.labels, conf if conf is not None else w.conf_logits,
                             workspace=self.ws, out=self.out, stream=stream)

    def parts(self):
        return [("stats", self.stats)]

    def bytes(self):
        w = self.w
        return {"stats": 2 * w.N * w.gamma * w.V * 4 + w.N * w.gamma * 16 + w.N * 8 + 64}

    def flops(self):
        return {}

    def e2e_compute(self, stream, dev_inputs, host_outputs):
        self.stats(stream, *dev_inputs)
        for h, d in zip(host_outputs, self.outputs()):
            h.copy_(d, non_blocking=True)

    def outputs(self):
        return [self.out["loss_num"], self.out["report"], self.out["num_tokens"], self.out["tau"]]

    def check(self):
        assert int((self.out["status"] != 0).sum()) == 0

    def cpu_sample(self, budget_s, max_requests=None):
        import oracle
        oracle.build()
        w = self.w
        done, n, t0 = 0, 0, time.perf_counter()
        while True:
            sl = slice(n, n + 1)
            oracle.accept_stats(synth.host(w.draft[sl]), synth.host(w.target[sl]), w.labels[sl].cpu().numpy(),
                                w.conf_logits[sl].cpu().numpy())
            done += 1
            n = (n + 1) % w.N
            el = time.perf_counter() - t0
            if el >= budget_s or (max_requests and done >= max_requests):
                break
        pos = done * w.gamma
        return {"value": pos / el, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{done} whole blocks ({pos} row pairs) of a {w.N}-block draw of the workload's "
                          f"recipe in {el:.1f} s, single-threaded C++ oracle"}


class StatsGrad(Stats):
    """The gradient of the statistics' loss numerators for one batch of row
    pairs: the draft-logit gradient rows written in full (they stay on the
    device for the optimizer; the end-to-end leg reads back the confidence
    gradients)."""

    def __init__(self, w, blocks=None):
        super().__init__(w, blocks)
        self.name = "training_stats_grad"

    def setup(self, ds, dev):
        w = self.w
        self.ds = ds
        N, g, V = w.N, w.gamma, w.V
        self.grads = (torch.empty((N, g, V), dtype=torch.float32, device=dev),
                      torch.empty((N, g), dtype=torch.float32, device=dev))
        self.inputs = [w.draft, w.target, w.labels, w.conf_logits]

    def stats(self, stream, draft=None, target=None, labels=None, conf=None):
        w = self.w
        self.ds.accept_stats_grad(draft if draft is not None else w.draft,
                                  target if target is not None else w.target,
                                  labels if labels is not None else w.labels,
                                  conf if conf is not None else w.conf_logits,
                                  scale=1.0, out=self.grads, stream=stream)

    def parts(self):
        return [("stats_grad", self.stats)]

    def bytes(self):
        w = self.w
        return {"stats_grad": 3 * w.N * w.gamma * w.V * 4 + w.N * w.gamma * 12}

    def outputs(self):
        return [self.grads[1]]

    def check(self):
        assert bool(torch.isfinite(self.grads[1]).all())

    def cpu_sample(self, budget_s, max_requests=None):
        import oracle
        oracle.build()
        w = self.w
        done, n, t0 = 0, 0, time.perf_counter()
        while True:
            sl = slice(n, n + 1)
            oracle.accept_stats_backward(synth.host(w.draft[sl]), synth.host(w.target[sl]),
                                         w.labels[sl].cpu().numpy(), w.conf_logits[sl].cpu().numpy())
            done += 1
            n = (n + 1) % w.N
            el = time.perf_counter() - t0
            if el >= budget_s or (max_requests and done >= max_requests):
                break
        pos = done * w.gamma
        return {"value": pos / el, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{done} whole blocks ({pos} row pairs) of a {w.N}-block draw of the workload's "
                          f"recipe in {el:.1f} s, single-threaded C++ oracle (gradient)"}


class StsFit:
    """Sequential Temperature Scaling of one serving log: a whole fit (every
    pass the device search takes) per step."""

    def __init__(self, log, blocks=None):
        self.log = log
        self.name = "sts_fit"
        self.positions = log.N * log.gamma  # pairs
        self.blocks = blocks or log.N

    def config(self):
        lg = self.log
        return {"workload": self.name, "blocks": self.blocks, "gamma": lg.gamma, "pairs": self.blocks * lg.gamma,
                "labels": "0/1 acceptances drawn from a miscalibrated confidence (T 0.6..3 over positions)",
                "mask": "90 % of the pairs counted"}

    def setup(self, ds, dev):
        lg = self.log
        self.ds = ds
        self.ws = ds.Workspace()
        self.out = (torch.empty((lg.gamma,), dtype=torch.float64, device=dev),
                    torch.empty((lg.gamma,), dtype=torch.int32, device=dev),
                    torch.empty((lg.gamma,), dtype=torch.int32, device=dev))
        self.inputs = [lg.conf_logits, lg.labels, lg.mask]

    def fit(self, stream, z=None, a=None, m=None):
        lg = self.log
        self.ds.sts_fit(z if z is not None else lg.conf_logits, a if a is not None else lg.labels,
                        m if m is not None else lg.mask, workspace=self.ws, out=self.out, stream=stream)

    def parts(self):
        return [("sts_fit", self.fit)]

    def bytes(self):
        """Every pass reads each pair once (z, a: 4 B each; the mask byte)
        until the last position stops: the largest passes count."""
        return {"sts_fit": int(self.out[2].max()) * self.positions * 9 + 64}

    def flops(self):
        return {}

    def e2e_compute(self, stream, dev_inputs, host_outputs):
        self.fit(stream, *dev_inputs)
        for h, d in zip(host_outputs, self.outputs()):
            h.copy_(d, non_blocking=True)

    def outputs(self):
        return [self.out[0], self.out[1]]

    def check(self):
        assert int((self.out[1] != 0).sum()) == 0, "a position of the benchmark log did not fit"

    def cpu_sample(self, budget_s, max_requests=None):
        """The oracle's fit on chunks of 4096 blocks of the log, one after the
        other, single-threaded."""
        import oracle
        oracle.build()
        lg = self.log
        chunk = min(4096, lg.N)
        z, a, m = (lg.conf_logits.cpu().numpy(), lg.labels.cpu().numpy(), lg.mask.cpu().numpy())
        done, n0, t0 = 0, 0, time.perf_counter()
        while True:
            sl = slice(n0, n0 + chunk)
            oracle.sts_fit(z[sl], a[sl], m[sl])
            done += 1
            n0 = (n0 + chunk) % max(1, lg.N - chunk + 1)
            el = time.perf_counter() - t0
            if el >= budget_s or (max_requests and done >= max_requests):
                break
        pairs = done * chunk * lg.gamma
        return {"value": pairs / el, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{done} fits of {chunk} blocks x {lg.gamma} pairs ({pairs} pairs) in {el:.1f} s, "
                          f"single-threaded C++ oracle (bisection)"}


def make_workload(name, device, stats_blocks=4096):
    if name == "full_decode_tile":
        return Serving(name, synth.full_decode_tile(device=device), 2)
    if name == "decode_verify_tile":
        return Serving(name, synth.decode_verify_tile(device=device), 2)
    if name == "mixed_serving":
        return Serving(name, synth.mixed_serving(device=device), 2)
    if name == "rnn_decode_tile":
        w = synth.decode_verify_tile(device=device)
        gw = synth.gru_weights(w.weights.r, synth._gen(1009, "cpu"), "cpu")  # small: drawn on the host
        return Serving(name, w, 2, gru=synth.GruWeights(*(t.to(device) for t in (gw.Wi, gw.Wh, gw.bi, gw.bh))))
    if name == "sts_fit":
        return StsFit(synth.sts_log(device=device))
    if name == "decode_verify_tile_width":
        w = synth.decode_verify_tile(device=device)
        return Serving(name, w, 2, width=synth.verify_widths(w.B, w.gamma))
    if name == "training_stats":
        return Stats(synth.training_stats(device=device, N=stats_blocks))
    if name == "training_stats_grad":
        return StatsGrad(synth.training_stats(device=device, N=stats_blocks))
    raise ValueError(name)


WORKLOADS = ("full_decode_tile", "decode_verify_tile", "mixed_serving", "decode_verify_tile_width",
             "rnn_decode_tile", "training_stats", "training_stats_grad", "sts_fit")


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import verify_dspark_markov_gb300 as ds
    from verify_dspark_markov_gb300 import build
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    ds.load()

    wl = make_workload(args.workload, dev, args.stats_blocks)
    wl.setup(ds, dev)
    stream = torch.cuda.current_stream(dev)
    parts = wl.parts()

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_r = torch.ones(max(2 * l2, 256 << 20) // 8, dtype=torch.int64, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        torch.sum(flush_r, dim=0, out=flush_sink)  # evict L2 by reading another 2 x L2 buffer

    # clock samples cover the warm-up, the timed steps and the end-to-end
    # steps (a short timed region alone may fall between two samples)
    clk = Clocks(local, args.clocks_csv).__enter__()
    time.sleep(0.3)  # let the sampler start
    w0 = time.time()
    for _ in range(args.warmup):
        flush_l2()
        for _, fn in parts:
            fn(stream)
    torch.cuda.synchronize()
    wl.check()

    steps = args.steps
    if args.max_seconds:  # keep the timed region near a minute for the big workloads
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _, fn in parts:
            fn(stream)
        b.record(stream)
        b.synchronize()
        steps = max(3, min(steps, int(args.max_seconds / max(a.elapsed_time(b) * 1e-3, 1e-6))))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        flush_l2()
        ev[i][0].record(stream)
        for j, (_, fn) in enumerate(parts):
            fn(stream)
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    step_ms = [ev[i][0].elapsed_time(ev[i][-1]) for i in range(steps)]
    part_ms = {name: float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)]))
               for j, (name, _) in enumerate(parts)}
    ms = replica_step_ms(float(np.mean(step_ms)), world, dev)

    # ---- end to end through the public API: host inputs, copies included.
    # Serving steps run as a serving loop would: the next step's inputs are
    # copied from pinned host memory on a second stream, into the other of
    # two device buffers, while this step computes.  The training workloads
    # (tens of GB of inputs a step, copy-bound by two orders of magnitude)
    # copy and compute in turn on one stream: there, copies running beside
    # the HBM-bound kernels measured slower.  Every step's copies and result
    # reads are inside the timed region.
    pipelined = isinstance(wl, Serving)
    nbuf = 2 if pipelined else 1
    host_in = [t.cpu().pin_memory() for t in wl.inputs]
    dev_in = [[torch.empty_like(t) for t in wl.inputs] for _ in range(nbuf)]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in wl.outputs()] for _ in range(nbuf)]
    copy_stream = torch.cuda.Stream(dev) if pipelined else stream
    copied = [torch.cuda.Event() for _ in range(nbuf)]
    consumed = [torch.cuda.Event() for _ in range(nbuf)]

    def e2e_run(n, start=None):
        if start is not None and pipelined:
            copy_stream.wait_event(start)
        for i in range(n):
            s = i % nbuf
            if pipelined and i >= nbuf:  # the buffer's previous step has been computed
                copy_stream.wait_event(consumed[s])
            with torch.cuda.stream(copy_stream):
                for d, h in zip(dev_in[s], host_in):
                    d.copy_(h, non_blocking=True)
                copied[s].record(copy_stream)
            stream.wait_event(copied[s])
            wl.e2e_compute(stream, dev_in[s], host_out[s])
            consumed[s].record(stream)

    e2e_run(2)
    torch.cuda.synchronize()
    n_e2e = max(3, min(20, steps // 10))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    e2e_run(n_e2e, start=a)
    b.record(stream)
    b.synchronize()
    torch.cuda.synchronize()
    e2e_ms = [a.elapsed_time(b) / n_e2e]
    w1 = time.time()
    time.sleep(0.1)
    clk.__exit__(None, None, None)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])

    hbm, tflops_peak, peak_kind = peaks()
    nbytes = wl.bytes()
    flops = wl.flops()
    dom = max(part_ms, key=part_ms.get)
    achieved = nbytes[dom] / (part_ms[dom] * 1e-3) / 1e9
    fused = False
    if isinstance(wl, Serving) and wl.gru is None:
        w = wl.w
        n_draft = ds.markov_launches(ds.BF16, w.B, w.gamma, w.V, w.weights.r, policy=not wl.greedy_only,
                                     conf=w.h is not None)
        fused = w.weights.r > 0 and n_draft == 1 + (1 if w.h is not None else 0)
    rnn_fused = False
    if isinstance(wl, Serving) and wl.gru is not None:
        w = wl.w
        rnn_fused = ds.rnn_launches(ds.BF16, w.B, w.gamma, w.V, w.weights.r, conf=w.h is not None) == \
            1 + (1 if w.h is not None else 0)
    draft_kernel = ("markov_fused_kernel (bias GEMM, policy and draw of every position in one launch) + "
                    "confidence_kernel" if fused else
                    "markov_fused_kernel, RNN head (GRU cell, bias GEMM, policy and draw of every position in one "
                    "launch) + confidence_kernel" if rnn_fused else
                    "rnn_sample (gru_step_kernel, the hi and lo markov_bias_kernel products and "
                    "markov_step_kernel per position)" if isinstance(wl, Serving) and wl.gru is not None else
                    "markov_sample (markov_bias_kernel + markov_step_kernel per position)")
    kernel = {"full_decode_tile": "argmax_rows_kernel<bf16> (draft + verify launches)",
              "training_stats": "stats_pairs_kernel<f32> (+ stats_blocks_kernel, stats_total_kernel)",
              "training_stats_grad": "stats_grad_kernel<f32>",
              "sts_fit": "sts_fit_kernel (every pass and update in one cooperative launch)"}.get(
                  wl.name, {"draft": draft_kernel,
                            "verify": "verify_rows_kernel<bf16>" if getattr(wl, "width", None) is None
                            else "verify_rows_kernel<bf16, width>"}.get(dom, dom))
    if wl.name == "full_decode_tile":  # the same kernel serves both parts: average over both launches
        achieved = sum(nbytes.values()) / (sum(part_ms.values()) * 1e-3) / 1e9
    result = {
        "metric": METRIC,
        "value": replica_throughput(wl.positions, ms, world),
        "unit": UNIT,
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if isinstance(wl, (Stats, StsFit)) else "bf16",
        "data": "synthetic",
        "config": dict(wl.config(), l2="inputs larger than L2, plus a 2 x L2 read of another buffer "
                                       "before every step",
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "roofline": {"bound": "hbm", "kernel": kernel, "part": dom, "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "peak_kind": peak_kind, "traffic": None,
                     "bytes_per_step": sum(nbytes.values())},
        "parts_ms": part_ms,
        "parts_GBps": {k: nbytes[k] / (part_ms[k] * 1e-3) / 1e9 for k in part_ms},
        "e2e": {"value": wl.positions * world / (float(np.mean(e2e_ms)) * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": float(np.mean(e2e_ms)),
                "steps": n_e2e,
                "schedule": ("pipelined: each step's host-to-device input copies run on a second stream, into the "
                             "other of two device buffers, while the previous step computes") if pipelined else
                            "sequential: copies, the step and the result read in turn on one stream"},
        "clocks": dict(clk.summary(w0, w1), window="warm-up, timed and end-to-end steps"),
        "wall_s_timed_region": wall,
    }
    if flops.get("draft"):
        t = flops["draft"] / (part_ms["draft"] * 1e-3) / 1e12
        result["tensor"] = {"part": "draft (markov_fused_kernel, tcgen05)" if fused or rnn_fused else
                            "draft (markov_bias_kernel, tcgen05)", "achieved": t,
                            "peak": tflops_peak, "unit": "TFLOP/s", "frac": t / tflops_peak,
                            "note": "FLOPs of the bias GEMM (the RNN head: its hi and lo products) over the "
                                    "whole draft part's time"}
    if isinstance(wl, Serving):
        g = wl.w.gamma
        if wl.name == "full_decode_tile":
            launches = 2
        elif wl.gru is not None:  # the library's own count for the RNN draft, then the verify
            launches = ds.rnn_launches(ds.BF16, wl.w.B, g, wl.w.V, wl.w.weights.r, conf=wl.w.h is not None) + 1
        else:  # the library's own count for the draft, then the verify
            launches = n_draft + 1
    elif isinstance(wl, StsFit):  # init, the fit, the status check
        launches = 3
    else:  # the statistics: pairs + per-block + total kernels; the gradient: one kernel
        launches = 1 if isinstance(wl, StatsGrad) else 3
    result["gpu_launches"] = launches * steps
    traffic = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(traffic):
        with open(traffic) as f:
            tr = json.load(f).get(wl.name)
        if tr:
            result["roofline"]["traffic"] = tr
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = wl.cpu_sample(args.cpu_seconds)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return result if rank == 0 else None


# ------------------------------------------------------------ reference arm
def make_workload_small(name):
    """The workload generated on the CPU for the oracle-only reference arm
    (the training statistics for 64 of its 4096 blocks)."""
    if name == "training_stats":
        return Stats(synth.training_stats(device="cpu", N=64), blocks=4096)
    if name == "training_stats_grad":
        return StatsGrad(synth.training_stats(device="cpu", N=64), blocks=4096)
    if name == "sts_fit":
        return StsFit(synth.sts_log(device="cpu", N=65_536), blocks=4_194_304)
    return make_workload(name, "cpu")


def run_reference(args):
    """The CPU oracle, as it stands, on bounded samples of the workload."""
    rank, world, local = dist_env()
    if rank != 0:
        return None
    wl = make_workload_small(args.workload)
    for _ in range(args.warmup):
        wl.cpu_sample(0.0, max_requests=1)
    per, t_steps = [], []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        per.append(wl.cpu_sample(min(10.0, args.cpu_seconds), max_requests=4))
        t_steps.append(time.perf_counter() - t0)
    value = float(np.mean([r["value"] for r in per]))
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": float(np.mean(t_steps)) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": dict(wl.config(), parallelism="single CPU thread"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": per[-1]["sample"] + " per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="full_decode_tile", choices=WORKLOADS)
    ap.add_argument("--max-seconds", type=float, default=30.0,
                    help="cap on the timed region's GPU time (fewer steps for slow workloads)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the nvidia-smi samples of the timed region in this file")
    ap.add_argument("--stats-blocks", type=int, default=4096,
                    help="training_stats only: blocks of the workload (smaller sizes for profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
