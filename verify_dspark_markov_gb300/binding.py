"""Thin ctypes binding of ``libdspark.so`` (the C ABI in ``include/dspark.h``).

Argument marshalling only: torch tensors supply device memory and the current
stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing or a CUDA device is absent,
the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

OK, EINVAL, ENOSPC, ECUDA, ENOTSUP = 0, -1, -2, -3, -4
BF16, F32 = 0, 1
OP_MARKOV_SAMPLE, OP_VERIFY, OP_ACCEPT_STATS, OP_STS_FIT, OP_RNN_SAMPLE = 0, 1, 2, 3, 4
REQ_OK, REQ_NONFINITE, REQ_EMPTY, REQ_TIMEOUT, REQ_BAD_POLICY, REQ_BAD_TOKEN = range(6)

EXPORTED = ("dspark_workspace_size", "dspark_markov_sample", "dspark_verify", "dspark_verify_width",
            "dspark_accept_stats", "dspark_accept_stats_grad", "dspark_status_string", "dspark_version",
            "dspark_verify_greedy_noalloc", "dspark_sts_fit", "dspark_rnn_sample", "dspark_markov_launches",
            "dspark_wait_selftest", "dspark_rnn_launches")

_lock = threading.Lock()
_lib = None


class DsparkError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load (but never build) the CUDA library; raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with "
                                   "verify_dspark_markov_gb300.build.build() first")
            lib = ctypes.CDLL(p)
            P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.dspark_workspace_size.argtypes = [i32] * 6
            lib.dspark_workspace_size.restype = sz
            lib.dspark_markov_sample.argtypes = ([P, i32, P, P, P, i32, P, i32, P, P, i32]
                                                 + [P] * 4 + [i32] * 3 + [P] * 6 + [sz, P])
            lib.dspark_markov_sample.restype = i32
            lib.dspark_verify.argtypes = [P, i32, P, P, P, P, P, P, P] + [i32] * 3 + [P] * 4 + [sz, P]
            lib.dspark_verify.restype = i32
            lib.dspark_verify_width.argtypes = ([P, i32, P, P, P, P, P, P, P, P] + [i32] * 3 + [P] * 4
                                                + [sz, P])
            lib.dspark_verify_width.restype = i32
            lib.dspark_accept_stats.argtypes = ([P, P, i32, P, P, P] + [i32] * 3 + [P] * 8
                                                + [sz, P])
            lib.dspark_accept_stats.restype = i32
            lib.dspark_accept_stats_grad.argtypes = ([P, P, i32, P, P, P] + [i32] * 3
                                                     + [ctypes.c_double, P, P, P])
            lib.dspark_accept_stats_grad.restype = i32
            lib.dspark_rnn_sample.argtypes = ([P, i32, P, P, P, i32, P, P, P, P, P, i32, P, P, i32]
                                              + [P] * 4 + [i32] * 3 + [P] * 6 + [sz, P])
            lib.dspark_rnn_sample.restype = i32
            lib.dspark_sts_fit.argtypes = [P, P, P, i32, i32, P, P, P, i32, P, sz, P]
            lib.dspark_sts_fit.restype = i32
            lib.dspark_status_string.argtypes = [i32]
            lib.dspark_status_string.restype = ctypes.c_char_p
            lib.dspark_wait_selftest.argtypes = [i32, i32, i32, P, P, P, P]
            lib.dspark_wait_selftest.restype = i32
            lib.dspark_rnn_launches.argtypes = [i32] * 6
            lib.dspark_rnn_launches.restype = i32
            lib.dspark_markov_launches.argtypes = [i32] * 7
            lib.dspark_markov_launches.restype = i32
            lib.dspark_version.argtypes = []
            lib.dspark_version.restype = i32
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().dspark_status_string(int(code)).decode()


def workspace_size(op: int, B: int, gamma: int, V: int, r: int = 0, H: int = 0) -> int:
    return int(load().dspark_workspace_size(op, B, gamma, V, r, H))


def wait_selftest(blocks: int, missing: int, limit_us: int, device=None, stream=None):
    """Blocks meeting at the library's bounded grid barrier, told to expect
    `missing` more arrivals than they make.  Returns (status int32 [blocks],
    waited_ns int64 [blocks]) on the device."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    status = torch.empty((blocks,), dtype=torch.int32, device=dev)
    waited = torch.empty((blocks,), dtype=torch.int64, device=dev)
    ws = torch.empty((256,), dtype=torch.uint8, device=dev)  # set by the call itself
    _check(load().dspark_wait_selftest(blocks, missing, limit_us, _ptr(status), _ptr(waited), _ptr(ws),
                                       _stream(stream)), "dspark_wait_selftest")
    if stream is not None:  # the buffer is in use on that stream until the kernels finish
        ws.record_stream(stream)
    return status, waited


def rnn_launches(dtype: int, B: int, gamma: int, V: int, r: int, conf: bool = False) -> int:
    """Kernels one rnn_sample call with these sizes enqueues on the current device."""
    n = int(load().dspark_rnn_launches(dtype, B, gamma, V, r, int(bool(conf))))
    if n < 0:
        raise ValueError("invalid sizes")
    return n


def markov_launches(dtype: int, B: int, gamma: int, V: int, r: int = 0, policy: bool = True,
                    conf: bool = False) -> int:
    """Kernels one markov_sample call with these sizes enqueues on the current device."""
    n = int(load().dspark_markov_launches(dtype, B, gamma, V, r, int(bool(policy)), int(bool(conf))))
    if n < 0:
        raise ValueError("invalid sizes")
    return n


# ------------------------------------------------------------------ helpers
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Workspace:
    """A zero-filled device buffer per (device, op); grown on demand.  The
    library leaves it zero-filled after every completed call."""

    def __init__(self):
        self._bufs = {}

    def get(self, op: int, nbytes: int, device) -> torch.Tensor | None:
        if nbytes == 0:
            return None
        key = (torch.device(device).index, op)
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(nbytes, dtype=torch.uint8, device=device)
            self._bufs[key] = buf
        return buf


_default_ws = Workspace()


def _check(code: int, what: str):
    if code != OK:
        raise DsparkError(code, what)


def _policy_ptr(policy):
    """policy: None (all greedy) or an int32 [B, 4] CUDA tensor of packed
    dspark_policy records (float temperature, int top_k, float top_p, int greedy)."""
    if policy is None:
        return None
    _dev(policy, "policy", torch.int32)
    if policy.dim() != 2 or policy.shape[1] != 4:
        raise ValueError("policy must be an int32 [B, 4] tensor of packed records")
    return _ptr(policy)


# ------------------------------------------------------------------ entry points
def rnn_sample(backbone, anchor, U, W, Wi, Wh, bi, bh, h=None, E=None, w_conf=None, policy=None,
               seed=None, request_id=None, pos0=None, workspace: Workspace | None = None, stream=None, out=None):
    """The draft's sequential head in its RNN form over [B, gamma, V] backbone
    logits: U, W bf16 [V, r]; Wi, Wh bf16 [3r, r] (gate rows r, z, n); bi, bh
    fp32 [3r].  Returns dict(proposals, q, q_at_x, conf, status) as
    markov_sample does."""
    _dev(backbone, "backbone")
    B, gamma, V = backbone.shape
    dev = backbone.device
    _dev(anchor, "anchor", torch.int32)
    for t, name in ((U, "U"), (W, "W"), (Wi, "Wi"), (Wh, "Wh")):
        _dev(t, name, torch.bfloat16)
    _dev(bi, "bi", torch.float32)
    _dev(bh, "bh", torch.float32)
    r = U.shape[1]
    if Wi.shape != (3 * r, r) or Wh.shape != (3 * r, r) or bi.shape != (3 * r,) or bh.shape != (3 * r,):
        raise ValueError("Wi, Wh must be [3r, r] and bi, bh [3r]")
    H, h_code = 0, F32
    if h is not None:
        _dev(h, "h")
        h_code = _dtype_code(h)
        H = h.shape[2]
        _dev(E, "E", torch.bfloat16)
        _dev(w_conf, "w_conf", torch.float32)
    if out is None:
        out = dict(proposals=torch.empty((B, gamma), dtype=torch.int32, device=dev),
                   q=(torch.empty((B, gamma, V), dtype=torch.float32, device=dev)
                      if policy is not None else None),
                   q_at_x=torch.empty((B, gamma), dtype=torch.float32, device=dev),
                   conf=(torch.empty((B, gamma), dtype=torch.float32, device=dev)
                         if h is not None else None),
                   status=torch.empty((B,), dtype=torch.int32, device=dev))
    ws_n = workspace_size(OP_RNN_SAMPLE, B, gamma, V, r, H)
    ws = (workspace or _default_ws).get(OP_RNN_SAMPLE, ws_n, dev)
    code = load().dspark_rnn_sample(
        _ptr(backbone), _dtype_code(backbone), _ptr(anchor), _ptr(U), _ptr(W), r, _ptr(Wi), _ptr(Wh), _ptr(bi),
        _ptr(bh), _ptr(h), h_code, _ptr(E), _ptr(w_conf), H, _policy_ptr(policy),
        _ptr(_dev(seed, "seed", torch.int64)), _ptr(_dev(request_id, "request_id", torch.int64)),
        _ptr(_dev(pos0, "pos0", torch.int64)), B, gamma, V, _ptr(out["proposals"]), _ptr(out["q"]),
        _ptr(out["q_at_x"]), _ptr(out["conf"]), _ptr(out["status"]), _ptr(ws), ws_n, _stream(stream))
    _check(code, "dspark_rnn_sample")
    return out


def verify(target, proposals, q=None, q_at_x=None, policy=None, seed=None, request_id=None,
           pos0=None, out=None, workspace: Workspace | None = None, stream=None, width=None):
    """Exact verify of [B, gamma+1, V] target logits against [B, gamma]
    proposals.  Returns (out_tokens [B, gamma+1], num_accepted [B], status [B]).
    width: None, or an int32 [B] CUDA tensor of per-request verify widths
    (0..gamma proposals checked; dspark_verify_width)."""
    _dev(target, "target")
    B, rows, V = target.shape
    gamma = rows - 1
    _dev(proposals, "proposals", torch.int32)
    if width is not None:
        _dev(width, "width", torch.int32)
        if width.shape != (B,):
            raise ValueError(f"width must have shape ({B},), got {tuple(width.shape)}")
    dev = target.device
    if out is None:
        out = (torch.empty((B, rows), dtype=torch.int32, device=dev),
               torch.empty((B,), dtype=torch.int32, device=dev),
               torch.empty((B,), dtype=torch.int32, device=dev))
    # greedy calls (policy None) keep their state on chip and take no workspace
    ws_n = workspace_size(OP_VERIFY, B, gamma, V) if policy is not None else 0
    ws = (workspace or _default_ws).get(OP_VERIFY, ws_n, dev)
    args = [_ptr(target), _dtype_code(target), _ptr(proposals), _ptr(_dev(q, "q", torch.float32)),
            _ptr(_dev(q_at_x, "q_at_x", torch.float32)), _policy_ptr(policy),
            _ptr(_dev(seed, "seed", torch.int64)), _ptr(_dev(request_id, "request_id", torch.int64)),
            _ptr(_dev(pos0, "pos0", torch.int64))]
    tail = [B, gamma, V, _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), _ptr(ws), ws_n, _stream(stream)]
    if width is None:
        code, what = load().dspark_verify(*args, *tail), "dspark_verify"
    else:
        code, what = load().dspark_verify_width(*args, _ptr(width), *tail), "dspark_verify_width"
    _check(code, what)
    return out


def markov_sample(backbone, anchor, U=None, W=None, h=None, E=None, w_conf=None, policy=None,
                  seed=None, request_id=None, pos0=None, workspace: Workspace | None = None,
                  stream=None, out=None):
    """The draft's sequential head over [B, gamma, V] backbone logits.
    Returns dict(proposals, q, q_at_x, conf, status)."""
    _dev(backbone, "backbone")
    B, gamma, V = backbone.shape
    dev = backbone.device
    _dev(anchor, "anchor", torch.int32)
    r = 0 if U is None else U.shape[1]
    if r:
        _dev(U, "U", torch.bfloat16)
        _dev(W, "W", torch.bfloat16)
    H = 0
    h_code = F32
    if h is not None:
        _dev(h, "h")
        h_code = _dtype_code(h)
        H = h.shape[2]
        _dev(E, "E", torch.bfloat16)
        _dev(w_conf, "w_conf", torch.float32)
    if out is None:
        out = dict(proposals=torch.empty((B, gamma), dtype=torch.int32, device=dev),
                   q=(torch.empty((B, gamma, V), dtype=torch.float32, device=dev)
                      if policy is not None else None),
                   q_at_x=torch.empty((B, gamma), dtype=torch.float32, device=dev),
                   conf=(torch.empty((B, gamma), dtype=torch.float32, device=dev)
                         if h is not None else None),
                   status=torch.empty((B,), dtype=torch.int32, device=dev))
    ws_n = workspace_size(OP_MARKOV_SAMPLE, B, gamma, V, r, H) if (policy is not None or r) else 0
    ws = (workspace or _default_ws).get(OP_MARKOV_SAMPLE, ws_n, dev)
    code = load().dspark_markov_sample(
        _ptr(backbone), _dtype_code(backbone), _ptr(anchor), _ptr(U), _ptr(W), r, _ptr(h), h_code,
        _ptr(E), _ptr(w_conf), H, _policy_ptr(policy),
        _ptr(_dev(seed, "seed", torch.int64)), _ptr(_dev(request_id, "request_id", torch.int64)),
        _ptr(_dev(pos0, "pos0", torch.int64)), B, gamma, V,
        _ptr(out["proposals"]), _ptr(out["q"]), _ptr(out["q_at_x"]), _ptr(out["conf"]),
        _ptr(out["status"]), _ptr(ws), ws_n, _stream(stream))
    _check(code, "dspark_markov_sample")
    return out


def accept_stats(draft, target, labels, conf_logits, mask=None, workspace: Workspace | None = None,
                 stream=None, out=None):
    """Acceptance statistics of [N, gamma, V] draft logits against the
    target.  Returns dict(l1, accept, tau, loss_num, report, num_tokens, status)."""
    _dev(draft, "draft")
    _dev(target, "target")
    if draft.shape != target.shape or draft.dtype != target.dtype:
        raise ValueError("draft and target must match in shape and dtype")
    N, gamma, V = draft.shape
    dev = draft.device
    _dev(labels, "labels", torch.int32)
    _dev(conf_logits, "conf_logits", torch.float32)
    _dev(mask, "mask", torch.uint8)
    if out is None:
        out = dict(l1=torch.empty((N, gamma), dtype=torch.float32, device=dev),
                   accept=torch.empty((N, gamma), dtype=torch.float32, device=dev),
                   tau=torch.empty((N,), dtype=torch.float32, device=dev),
                   loss_num=torch.empty((4,), dtype=torch.float64, device=dev),
                   report=torch.empty((2,), dtype=torch.float64, device=dev),
                   num_tokens=torch.empty((1,), dtype=torch.int64, device=dev),
                   status=torch.empty((N,), dtype=torch.int32, device=dev))
    ws_n = workspace_size(OP_ACCEPT_STATS, N, gamma, V)
    ws = (workspace or _default_ws).get(OP_ACCEPT_STATS, ws_n, dev)
    code = load().dspark_accept_stats(
        _ptr(draft), _ptr(target), _dtype_code(draft), _ptr(labels), _ptr(conf_logits), _ptr(mask),
        N, gamma, V, _ptr(out["l1"]), _ptr(out["accept"]), _ptr(out["tau"]), _ptr(out["loss_num"]),
        _ptr(out["report"]), _ptr(out["num_tokens"]), _ptr(out["status"]), _ptr(ws), ws_n,
        _stream(stream))
    _check(code, "dspark_accept_stats")
    return out


def accept_stats_grad(draft, target, labels, conf_logits, mask=None, scale=1.0, stream=None, out=None):
    """Gradient of the statistics' loss 0.1 CE + 0.9 L1 + 1.0 BCE (weighted,
    masked numerators; target and the BCE label held fixed) with respect to
    the draft logits and the confidence logits, times scale.  Returns
    (grad_draft fp32 [N, gamma, V], grad_conf fp32 [N, gamma])."""
    _dev(draft, "draft")
    _dev(target, "target")
    if draft.shape != target.shape or draft.dtype != target.dtype:
        raise ValueError("draft and target must match in shape and dtype")
    N, gamma, V = draft.shape
    dev = draft.device
    _dev(labels, "labels", torch.int32)
    _dev(conf_logits, "conf_logits", torch.float32)
    _dev(mask, "mask", torch.uint8)
    if out is None:
        out = (torch.empty((N, gamma, V), dtype=torch.float32, device=dev),
               torch.empty((N, gamma), dtype=torch.float32, device=dev))
    code = load().dspark_accept_stats_grad(
        _ptr(draft), _ptr(target), _dtype_code(draft), _ptr(labels), _ptr(conf_logits), _ptr(mask),
        N, gamma, V, float(scale), _ptr(out[0]), _ptr(out[1]), _stream(stream))
    _check(code, "dspark_accept_stats_grad")
    return out


def sts_fit(conf_logits, labels, mask=None, max_passes=0, workspace: Workspace | None = None, stream=None,
            out=None):
    """Sequential Temperature Scaling: per block position the inverse
    temperature beta >= 0 of the confidence head, from fp32 [N, gamma]
    confidence logits and accept labels (mask: uint8 [N, gamma] or None);
    max_passes is the pass budget (0: the library's default).
    Returns (beta float64 [gamma], status int32 [gamma], passes int32
    [gamma]: the passes each position's search used)."""
    _dev(conf_logits, "conf_logits", torch.float32)
    _dev(labels, "labels", torch.float32)
    if conf_logits.dim() != 2 or labels.shape != conf_logits.shape:
        raise ValueError("conf_logits and labels must be [N, gamma] tensors of one shape")
    N, gamma = conf_logits.shape
    if mask is not None:
        _dev(mask, "mask", torch.uint8)
        if mask.shape != conf_logits.shape:
            raise ValueError("mask must have the shape of conf_logits")
    dev = conf_logits.device
    if out is None:
        out = (torch.empty((gamma,), dtype=torch.float64, device=dev),
               torch.empty((gamma,), dtype=torch.int32, device=dev),
               torch.empty((gamma,), dtype=torch.int32, device=dev))
    ws_n = workspace_size(OP_STS_FIT, N, gamma, 8)
    ws = (workspace or _default_ws).get(OP_STS_FIT, ws_n, dev)
    code = load().dspark_sts_fit(_ptr(conf_logits), _ptr(labels), _ptr(mask), N, gamma, _ptr(out[0]),
                                 _ptr(out[1]), _ptr(out[2]), int(max_passes), _ptr(ws), ws_n, _stream(stream))
    _check(code, "dspark_sts_fit")
    return out
