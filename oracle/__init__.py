"""ORACLE - test infrastructure, not product code.

Builds the plain C++ oracle (``dspark_oracle.cpp``) with the host compiler and
exposes it to Python through ctypes with numpy arrays.  Only the test suite,
``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` / reference
leg may import this package; the CUDA library never does.

Each function follows the passage cited in ``dspark_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.cpp")
_HDR = os.path.join(_HERE, "dspark_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libdspark_oracle.so")

_lock = threading.Lock()
_lib = None

OK, NONFINITE, EMPTY, BAD_POLICY, BAD_TOKEN = 0, 1, 2, 4, 5
TOL = 1e-5


def build(force: bool = False) -> str:
    """Compile the oracle to ``oracle/_build/libdspark_oracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= newest_src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, u32, f32, f64 = ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_double
            lib.orc_philox4x32_10.argtypes = [u32, u32, P, P]
            lib.orc_philox4x32_10.restype = None
            lib.orc_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, u32]
            lib.orc_uniform.restype = f64
            lib.orc_policy_row.argtypes = [P, i32, f32, i32, f32, i32, i32, P, P, P, P]
            lib.orc_policy_row.restype = i32
            lib.orc_sample_index.argtypes = [P, i32, f64, P]
            lib.orc_sample_index.restype = i32
            lib.orc_markov_sample.argtypes = ([P, i32, P, P, P, i32, P, i32, P, P, i32]
                                              + [P] * 7 + [i32, i32, i32] + [P] * 6)
            lib.orc_markov_sample.restype = None
            lib.orc_rnn_sample.argtypes = ([P, i32, P, P, P, i32, P, P, P, P, P, i32, P, P, i32]
                                           + [P] * 7 + [i32] * 3 + [P] * 7)
            lib.orc_rnn_sample.restype = None
            lib.orc_sts_fit.argtypes = [P, P, P, i32, i32, P, P]
            lib.orc_sts_fit.restype = None
            lib.orc_verify.argtypes = [P, i32, P, P, P] + [P] * 7 + [i32, i32, i32] + [P] * 6
            lib.orc_verify.restype = None
            lib.orc_verify_width.argtypes = [P, i32, P, P, P] + [P] * 7 + [i32, i32, i32] + [P] * 7
            lib.orc_verify_width.restype = None
            lib.orc_accept_stats.argtypes = [P, P, i32, P, P, P, i32, i32, i32] + [P] * 7
            lib.orc_accept_stats.restype = None
            lib.orc_accept_stats_backward.argtypes = [P, P, i32, P, P, P, i32, i32, i32, f64, P, P]
            lib.orc_accept_stats_backward.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dtype_code(arr: np.ndarray) -> int:
    """0 = bf16 (stored as uint16 bit patterns), 1 = fp32."""
    if arr.dtype == np.uint16:
        return 0
    if arr.dtype == np.float32:
        return 1
    raise TypeError(f"logits must be uint16 (bf16 bits) or float32, got {arr.dtype}")


# ----------------------------------------------------------------- primitives
def philox4x32_10(key0: int, key1: int, ctr) -> np.ndarray:
    c = _c(ctr, np.uint32)
    out = np.zeros(4, np.uint32)
    _load().orc_philox4x32_10(key0 & 0xFFFFFFFF, key1 & 0xFFFFFFFF, _ptr(c), _ptr(out))
    return out


def uniform(seed: int, request_id: int, pos: int, draw: int) -> float:
    return _load().orc_uniform(seed, request_id, pos, draw)


def policy_row(z, temperature=1.0, top_k=0, top_p=1.0, greedy=False, exact_logits=True):
    """Returns (status, p[V] float64, argmax, support_size, indeterminate)."""
    z = _c(z, np.float64)
    p = np.zeros(z.shape[0], np.float64)
    am, sup, ind = (np.zeros(1, np.int32) for _ in range(3))
    st = _load().orc_policy_row(_ptr(z), z.shape[0], float(temperature), int(top_k),
                                float(top_p), int(bool(greedy)), int(bool(exact_logits)),
                                _ptr(p), _ptr(am), _ptr(sup), _ptr(ind))
    return st, p, int(am[0]), int(sup[0]), bool(ind[0])


def sample_index(w, u: float):
    w = _c(w, np.float64)
    margin = np.zeros(1, np.float64)
    i = _load().orc_sample_index(_ptr(w), w.shape[0], float(u), _ptr(margin))
    return int(i), float(margin[0])


# ------------------------------------------------------------------ the path
def _policy_arrays(policy):
    """policy: dict of per-request arrays temperature/top_k/top_p/greedy."""
    return (_c(policy["temperature"], np.float32), _c(policy["top_k"], np.int32),
            _c(policy["top_p"], np.float32), _c(policy["greedy"], np.int32))


def markov_sample(backbone, anchor, U, W, h, E, w_conf, policy, seed, request_id, pos0):
    """backbone [B,gamma,V] (uint16 bf16 bits or float32); U, W uint16 [V,r]
    (r may be 0); h [B,gamma,H] or None; E uint16 [V,H]; w_conf float32 [2H].
    Returns dict(proposals, q, q_at_x, conf, status, indet)."""
    backbone = np.ascontiguousarray(backbone)
    B, gamma, V = backbone.shape
    anchor = _c(anchor, np.int32)
    r = 0 if U is None else U.shape[1]
    Uc = _c(U, np.uint16) if r else None
    Wc = _c(W, np.uint16) if r else None
    T, K, P, G = _policy_arrays(policy)
    H = 0
    hc = Ec = wc = None
    h_dtype = 1
    if h is not None:
        hc = np.ascontiguousarray(h)
        h_dtype = _dtype_code(hc)
        H = hc.shape[2]
        Ec = _c(E, np.uint16)
        wc = _c(w_conf, np.float32)
    seed = _c(seed, np.uint64)
    rid = _c(request_id, np.uint64)
    p0 = _c(pos0, np.int64)
    proposals = np.full((B, gamma), -7, np.int32)
    q = np.zeros((B, gamma, V), np.float32)
    q_at_x = np.zeros((B, gamma), np.float32)
    conf = np.zeros((B, gamma), np.float32) if h is not None else None
    status = np.zeros(B, np.int32)
    indet = np.zeros((B, gamma), np.uint8)
    _load().orc_markov_sample(_ptr(backbone), _dtype_code(backbone), _ptr(anchor), _ptr(Uc),
                              _ptr(Wc), r, _ptr(hc), h_dtype, _ptr(Ec), _ptr(wc), H,
                              _ptr(T), _ptr(K), _ptr(P), _ptr(G), _ptr(seed), _ptr(rid),
                              _ptr(p0), B, gamma, V, _ptr(proposals), _ptr(q), _ptr(q_at_x),
                              _ptr(conf), _ptr(status), _ptr(indet))
    return dict(proposals=proposals, q=q, q_at_x=q_at_x, conf=conf, status=status,
                indet=indet.astype(bool))


def rnn_sample(backbone, anchor, U, W, Wi, Wh, bi, bh, h, E, w_conf, policy, seed, request_id, pos0):
    """The RNN-head sampler: as markov_sample, plus the GRU weights Wi, Wh
    uint16 [3r, r] (bf16 bits; gate order r, z, n) and bi, bh float32 [3r].
    Returns markov_sample's dict plus states float64 [B, gamma, r]."""
    backbone = np.ascontiguousarray(backbone)
    B, gamma, V = backbone.shape
    anchor = _c(anchor, np.int32)
    r = U.shape[1]
    Uc, Wc = _c(U, np.uint16), _c(W, np.uint16)
    Wic, Whc = _c(Wi, np.uint16), _c(Wh, np.uint16)
    bic, bhc = _c(bi, np.float32), _c(bh, np.float32)
    assert Wic.shape == (3 * r, r) and Whc.shape == (3 * r, r) and bic.shape == (3 * r,) and bhc.shape == (3 * r,)
    T, K, P, G = _policy_arrays(policy)
    H = 0
    hc = Ec = wc = None
    h_dtype = 1
    if h is not None:
        hc = np.ascontiguousarray(h)
        h_dtype = _dtype_code(hc)
        H = hc.shape[2]
        Ec = _c(E, np.uint16)
        wc = _c(w_conf, np.float32)
    seed = _c(seed, np.uint64)
    rid = _c(request_id, np.uint64)
    p0 = _c(pos0, np.int64)
    proposals = np.full((B, gamma), -7, np.int32)
    q = np.zeros((B, gamma, V), np.float32)
    q_at_x = np.zeros((B, gamma), np.float32)
    conf = np.zeros((B, gamma), np.float32) if h is not None else None
    status = np.zeros(B, np.int32)
    indet = np.zeros((B, gamma), np.uint8)
    states = np.zeros((B, gamma, r), np.float64)
    _load().orc_rnn_sample(_ptr(backbone), _dtype_code(backbone), _ptr(anchor), _ptr(Uc), _ptr(Wc), r,
                           _ptr(Wic), _ptr(Whc), _ptr(bic), _ptr(bhc), _ptr(hc), h_dtype, _ptr(Ec), _ptr(wc), H,
                           _ptr(T), _ptr(K), _ptr(P), _ptr(G), _ptr(seed), _ptr(rid), _ptr(p0), B, gamma, V,
                           _ptr(proposals), _ptr(q), _ptr(q_at_x), _ptr(conf), _ptr(status), _ptr(indet),
                           _ptr(states))
    return dict(proposals=proposals, q=q, q_at_x=q_at_x, conf=conf, status=status,
                indet=indet.astype(bool), states=states)


def verify(target, proposals, q, q_at_x, policy, seed, request_id, pos0, width=None):
    """target [B,gamma+1,V] (uint16 bf16 bits or float32); proposals int32
    [B,gamma]; q float32 [B,gamma,V] or None (all-greedy batch); q_at_x float32
    [B,gamma] or None; width int32 [B] (proposals each request verifies,
    0..gamma) or None (all gamma).  Returns dict(out_tokens, num_accepted,
    status, indet, det_tokens, det_nacc): det_tokens [B] leading out_tokens
    entries decided before the request's first indeterminate decision,
    det_nacc [B] whether num_accepted was (all of it when indet is False)."""
    target = np.ascontiguousarray(target)
    B, rows, V = target.shape
    gamma = rows - 1
    x = _c(proposals, np.int32)
    qc = None if q is None else _c(q, np.float32)
    qx = np.ones((B, gamma), np.float32) if q_at_x is None else _c(q_at_x, np.float32)
    T, K, P, G = _policy_arrays(policy)
    if qc is None and not np.all(G != 0):
        raise ValueError("q is required for non-greedy requests")
    if qc is None:
        qc = np.zeros((1,), np.float32)
    seed = _c(seed, np.uint64)
    rid = _c(request_id, np.uint64)
    p0 = _c(pos0, np.int64)
    out = np.zeros((B, rows), np.int32)
    nacc = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    indet = np.zeros(B, np.uint8)
    det_tokens = np.zeros(B, np.int32)
    det_nacc = np.zeros(B, np.uint8)
    if width is None:
        _load().orc_verify(_ptr(target), _dtype_code(target), _ptr(x), _ptr(qc), _ptr(qx),
                           _ptr(T), _ptr(K), _ptr(P), _ptr(G), _ptr(seed), _ptr(rid), _ptr(p0),
                           B, gamma, V, _ptr(out), _ptr(nacc), _ptr(status), _ptr(indet),
                           _ptr(det_tokens), _ptr(det_nacc))
    else:
        wd = _c(width, np.int32)
        _load().orc_verify_width(_ptr(target), _dtype_code(target), _ptr(x), _ptr(qc), _ptr(qx),
                                 _ptr(T), _ptr(K), _ptr(P), _ptr(G), _ptr(seed), _ptr(rid), _ptr(p0),
                                 B, gamma, V, _ptr(wd), _ptr(out), _ptr(nacc), _ptr(status), _ptr(indet),
                                 _ptr(det_tokens), _ptr(det_nacc))
    return dict(out_tokens=out, num_accepted=nacc, status=status, indet=indet.astype(bool),
                det_tokens=det_tokens, det_nacc=det_nacc.astype(bool))


def accept_stats(draft, target, labels, conf_logits, mask=None):
    """draft, target [N,gamma,V] (uint16 bf16 bits or float32).  Returns
    dict(l1, accept, tau, loss_num[4], report[2], num_tokens, status)."""
    draft = np.ascontiguousarray(draft)
    target = np.ascontiguousarray(target)
    if draft.shape != target.shape or draft.dtype != target.dtype:
        raise ValueError("draft and target must match in shape and dtype")
    N, gamma, V = draft.shape
    y = _c(labels, np.int32)
    zc = _c(conf_logits, np.float32)
    m = None if mask is None else _c(mask, np.uint8)
    l1 = np.zeros((N, gamma), np.float32)
    acc = np.zeros((N, gamma), np.float32)
    tau = np.zeros(N, np.float32)
    loss = np.zeros(4, np.float64)
    report = np.zeros(2, np.float64)
    ntok = np.zeros(1, np.int64)
    status = np.zeros(N, np.int32)
    _load().orc_accept_stats(_ptr(draft), _ptr(target), _dtype_code(draft), _ptr(y), _ptr(zc),
                             _ptr(m), N, gamma, V, _ptr(l1), _ptr(acc), _ptr(tau), _ptr(loss),
                             _ptr(report), _ptr(ntok), _ptr(status))
    return dict(l1=l1, accept=acc, tau=tau, loss_num=loss, report=report,
                num_tokens=int(ntok[0]), status=status)


def accept_stats_backward(draft, target, labels, conf_logits, mask=None, scale=1.0):
    """Gradient of 0.1 CE + 0.9 L1 + 1.0 BCE (weighted, masked numerators)
    with respect to the draft logits and the confidence logits, the target
    and the BCE label held fixed, times scale.  Returns (grad_draft float32
    [N,gamma,V], grad_conf float32 [N,gamma])."""
    draft = np.ascontiguousarray(draft)
    target = np.ascontiguousarray(target)
    if draft.shape != target.shape or draft.dtype != target.dtype:
        raise ValueError("draft and target must match in shape and dtype")
    N, gamma, V = draft.shape
    y = _c(labels, np.int32)
    zc = _c(conf_logits, np.float32)
    m = None if mask is None else _c(mask, np.uint8)
    gd = np.zeros((N, gamma, V), np.float32)
    gc = np.zeros((N, gamma), np.float32)
    _load().orc_accept_stats_backward(_ptr(draft), _ptr(target), _dtype_code(draft), _ptr(y), _ptr(zc),
                                      _ptr(m), N, gamma, V, float(scale), _ptr(gd), _ptr(gc))
    return gd, gc


def sts_fit(conf_logits, labels, mask=None):
    """Sequential Temperature Scaling: conf_logits, labels float32 [N, gamma];
    mask uint8 [N, gamma] or None.  Returns dict(beta float64 [gamma],
    status int32 [gamma])."""
    z = _c(conf_logits, np.float32)
    a = _c(labels, np.float32)
    N, gamma = z.shape
    m = None if mask is None else _c(mask, np.uint8)
    beta = np.zeros(gamma, np.float64)
    status = np.zeros(gamma, np.int32)
    _load().orc_sts_fit(_ptr(z), _ptr(a), _ptr(m), N, gamma, _ptr(beta), _ptr(status))
    return dict(beta=beta, status=status)
