"""fp64 CPU oracle of the speculative-decoding verification step (ctypes wrapper).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU library in
``speculative_decoding_verification_top_gb300`` shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, no vectorisation);
this module only compiles it with gcc and marshals numpy arrays.  Logits are
passed in their storage dtype: ``np.float32`` arrays, or ``np.uint16``
arrays holding bf16 bit patterns; the C code upcasts each one exactly.

Status codes (the oracle's own numbering; names match the GPU library's):
a returned error word is the OR of ``1 << code`` over every failed check.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1
STOCHASTIC, GREEDY = 0, 1

ROW_NONFINITE = 1
ROW_ALL_NEG_INF = 2
TOKEN_RANGE = 3
UNIFORM_RANGE = 4
TREE_SHAPE = 5
PROB_RANGE = 6
CODE_NAMES = {
    ROW_NONFINITE: "ROW_NONFINITE",
    ROW_ALL_NEG_INF: "ROW_ALL_NEG_INF",
    TOKEN_RANGE: "TOKEN_RANGE",
    UNIFORM_RANGE: "UNIFORM_RANGE",
    TREE_SHAPE: "TREE_SHAPE",
    PROB_RANGE: "PROB_RANGE",
}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no -ffast-math)."""
    fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)
    if force or not fresh:
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I, D = ctypes.c_int, ctypes.c_double
        lib.oracle_process_row.argtypes = [P, I, I, D, D, P, P]
        lib.oracle_process_row.restype = I
        lib.oracle_process_row_k.argtypes = [P, I, I, D, D, I, P, P]
        lib.oracle_process_row_k.restype = I
        lib.oracle_verify_sample_k.argtypes = [P, P, I, P, P, I, I, I, D, D, I, I, P, P, P, P]
        lib.oracle_verify_sample_k.restype = I
        lib.oracle_verify_sample_probs_k.argtypes = [P, P, I, P, P, I, I, I, D, D, I, P, P, P, P]
        lib.oracle_verify_sample_probs_k.restype = I
        lib.oracle_acceptance_k.argtypes = [P, P, I, I, I, I, D, D, I, P, P]
        lib.oracle_acceptance_k.restype = I
        lib.oracle_argmax_row.argtypes = [P, I, I, P]
        lib.oracle_argmax_row.restype = I
        lib.oracle_inverse_cdf.argtypes = [P, I, D, P]
        lib.oracle_inverse_cdf.restype = ctypes.c_int32
        lib.oracle_verify_sample.argtypes = [P, P, I, P, P, I, I, I, D, D, I, P, P, P, P]
        lib.oracle_verify_sample.restype = I
        lib.oracle_verify_sample_probs.argtypes = [P, P, I, P, P, I, I, I, D, D, P, P, P, P]
        lib.oracle_verify_sample_probs.restype = I
        lib.oracle_acceptance.argtypes = [P, P, I, I, I, I, D, D, P, P]
        lib.oracle_acceptance.restype = I
        lib.oracle_tree_mask.argtypes = [P, P, I, I, P, P]
        lib.oracle_tree_mask.restype = I
        lib.oracle_ancestor_mask.argtypes = [P, I, P]
        lib.oracle_ancestor_mask.restype = I
        lib.oracle_verify_tree_sample.argtypes = [P, P, I, P, P, P, I, I, I, I, D, D, I, P, P, P, P]
        lib.oracle_verify_tree_sample.restype = I
        lib.oracle_verify_tree.argtypes = [P, I, P, P, I, I, I, I, P, P, P]
        lib.oracle_verify_tree.restype = I
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError("logits must be float32 or uint16 (bf16 bit patterns), got %s" % a.dtype)


def process_row(logits, T: float = 1.0, top_p: float = 1.0, top_k: int = 0):
    """Processed distribution of one row (temperature, top-k, then top-p).

    Returns (status, prob[V] float64, info[4]) with info = (Z, tau,
    mass above tau, mass at and above tau).
    """
    row, dt = _logits(logits)
    V = row.shape[-1]
    prob = np.zeros(V, np.float64)
    info = np.zeros(4, np.float64)
    st = _load().oracle_process_row_k(_ptr(row), dt, V, float(T), float(top_p), int(top_k),
                                      _ptr(prob), _ptr(info))
    return st, prob, info


def argmax_row(logits):
    row, dt = _logits(logits)
    out = np.zeros(1, np.int32)
    st = _load().oracle_argmax_row(_ptr(row), dt, row.shape[-1], _ptr(out))
    return st, int(out[0])


def inverse_cdf(w, u: float):
    """Inverse-CDF draw; returns (token, (S, C(token-1), C(token)))."""
    w = np.ascontiguousarray(w, np.float64)
    edges = np.zeros(3, np.float64)
    tok = _load().oracle_inverse_cdf(_ptr(w), w.shape[0], float(u), _ptr(edges))
    return int(tok), tuple(edges)


def verify_sample(target, draft, draft_tokens, uniforms, T=1.0, top_p=1.0, mode=STOCHASTIC,
                  debug=False, top_k=0):
    """One verification step for B sequences.

    target [B, k+1, V], draft [B, k, V] (None in GREEDY), draft_tokens [B, k]
    int32, uniforms [B, k+1] float32 (None in GREEDY).
    Returns dict(tokens [B, k+1], num_accepted [B], errors, and with
    debug=True: dbg [B, 2k+3] = P_1..P_k, Q_1..Q_k, S, C(tok-1), C(tok);
    row_info [B, 2k+1, 4]).
    """
    tgt, dt = _logits(target)
    B, k1, V = tgt.shape
    k = k1 - 1
    drf = None
    if draft is not None:
        drf, dt2 = _logits(draft)
        if dt2 != dt or drf.shape != (B, k, V):
            raise ValueError("draft logits must match target dtype and be [B, k, V]")
    toks = np.ascontiguousarray(draft_tokens, np.int32).reshape(B, k)
    uni = None if uniforms is None else np.ascontiguousarray(uniforms, np.float32).reshape(B, k + 1)
    out_t = np.zeros((B, k + 1), np.int32)
    out_n = np.zeros(B, np.int32)
    dbg = np.zeros((B, 2 * k + 3), np.float64) if debug else None
    R = 2 * k + 1 if mode == STOCHASTIC else k + 1
    info = np.zeros((B, R, 4), np.float64) if debug else None
    err = _load().oracle_verify_sample_k(
        _ptr(tgt), _ptr(drf), dt, _ptr(toks), _ptr(uni), B, k, V, float(T), float(top_p),
        int(top_k), int(mode), _ptr(out_t), _ptr(out_n), _ptr(dbg), _ptr(info))
    if err < 0:
        raise ValueError("oracle_verify_sample rejected its arguments")
    res = dict(tokens=out_t, num_accepted=out_n, errors=err)
    if debug:
        res.update(dbg=dbg, row_info=info)
    return res


def verify_sample_probs(target, draft_probs, draft_tokens, uniforms, T=1.0, top_p=1.0,
                        debug=False, top_k=0):
    """verify_sample with the draft given as probabilities: draft_probs
    [B, k, V] float32 is q itself (used as given; temperature and top-p
    process the target rows only).  Same results; with debug=True row_info
    is [B, k+1, 4] (target rows)."""
    tgt, dt = _logits(target)
    B, k1, V = tgt.shape
    k = k1 - 1
    q = np.ascontiguousarray(draft_probs, np.float32)
    if q.shape != (B, k, V):
        raise ValueError("draft_probs must be float32 [B, k, V]")
    toks = np.ascontiguousarray(draft_tokens, np.int32).reshape(B, k)
    uni = np.ascontiguousarray(uniforms, np.float32).reshape(B, k + 1)
    out_t = np.zeros((B, k + 1), np.int32)
    out_n = np.zeros(B, np.int32)
    dbg = np.zeros((B, 2 * k + 3), np.float64) if debug else None
    info = np.zeros((B, k + 1, 4), np.float64) if debug else None
    err = _load().oracle_verify_sample_probs_k(
        _ptr(tgt), _ptr(q), dt, _ptr(toks), _ptr(uni), B, k, V, float(T), float(top_p),
        int(top_k), _ptr(out_t), _ptr(out_n), _ptr(dbg), _ptr(info))
    if err < 0:
        raise ValueError("oracle_verify_sample_probs rejected its arguments")
    res = dict(tokens=out_t, num_accepted=out_n, errors=err)
    if debug:
        res.update(dbg=dbg, row_info=info)
    return res


def acceptance(target, draft, T=1.0, top_p=1.0, top_k=0):
    """Per-position acceptance rate beta [B, k] = sum_x min(p_i, q_i) and
    total-variation distance tv [B, k] = (1/2) sum_x |p_i - q_i|, each from
    its own definition.  target [B, k+1, V], draft [B, k, V].
    Returns dict(beta, tv, errors); NaN marks a pair with a data error."""
    tgt, dt = _logits(target)
    drf, dt2 = _logits(draft)
    B, k1, V = tgt.shape
    k = k1 - 1
    if dt2 != dt or drf.shape != (B, k, V):
        raise ValueError("draft logits must match target dtype and be [B, k, V]")
    beta = np.zeros((B, k), np.float64)
    tv = np.zeros((B, k), np.float64)
    err = _load().oracle_acceptance_k(_ptr(tgt), _ptr(drf), dt, B, k, V, float(T), float(top_p),
                                      int(top_k), _ptr(beta), _ptr(tv))
    if err < 0:
        raise ValueError("oracle_acceptance rejected its arguments")
    return dict(beta=beta, tv=tv, errors=err)


def ancestor_mask(parents):
    par = np.ascontiguousarray(parents, np.int32)
    N = par.shape[0]
    mask = np.zeros((N, N), np.uint8)
    st = _load().oracle_ancestor_mask(_ptr(par), N, _ptr(mask))
    return st, mask


def tree_mask(parents, pos0=None):
    """Tree attention mask [B, N, N] (uint8, 1 = may attend: self and
    ancestors) and positions [B, N] (pos0[b] + depth) for parents [B, N].
    Returns dict(mask, pos, errors)."""
    par = np.ascontiguousarray(parents, np.int32)
    B, N = par.shape
    p0 = None if pos0 is None else np.ascontiguousarray(pos0, np.int32).reshape(B)
    mask = np.zeros((B, N, N), np.uint8)
    pos = np.zeros((B, N), np.int32)
    err = _load().oracle_tree_mask(_ptr(par), _ptr(p0), B, N, _ptr(mask), _ptr(pos))
    if err < 0:
        raise ValueError("oracle_tree_mask rejected its arguments")
    return dict(mask=mask, pos=pos, errors=err)


def verify_tree(target, parents, node_tokens, depth):
    """Greedy tree verification; target [B, N, V], parents [N], node_tokens [B, N].

    Returns dict(tokens [B, D+1], num_accepted [B], path [B, D+1], errors).
    """
    tgt, dt = _logits(target)
    B, N, V = tgt.shape
    par = np.ascontiguousarray(parents, np.int32)
    tok = np.ascontiguousarray(node_tokens, np.int32).reshape(B, N)
    W = depth + 1
    out_t = np.zeros((B, W), np.int32)
    out_n = np.zeros(B, np.int32)
    out_p = np.zeros((B, W), np.int32)
    err = _load().oracle_verify_tree(_ptr(tgt), dt, _ptr(par), _ptr(tok), B, N, V, int(depth),
                                     _ptr(out_t), _ptr(out_n), _ptr(out_p))
    if err < 0:
        raise ValueError("oracle_verify_tree rejected its arguments")
    return dict(tokens=out_t, num_accepted=out_n, path=out_p, errors=err)


def boundary_kinds(res, uniforms, top_p=1.0, tol=1e-5):
    """Sequences whose outcome sits within `tol` of a decision boundary, by
    kind, as three boolean arrays [B]:

    accept  -- at an accept test the oracle ran, |u_i - P_i / Q_i| < tol
               (the accept count itself may differ in float32);
    cdf     -- at the final draw, |u - C(x-1)/S| or |u - C(x)/S| < tol at
               the drawn token x (only the drawn token may differ);
    nucleus -- (top-p) a row's cumulative mass before or at its threshold
               is within tol of top_p (its kept set, and with it any later
               quantity, may differ).

    Sequences the oracle rejected as invalid (num_accepted < 0) are never
    flagged.  `res` must come from verify_sample(..., debug=True).
    """
    dbg, info = res["dbg"], res["row_info"]
    B = dbg.shape[0]
    k = (dbg.shape[1] - 3) // 2
    u = np.asarray(uniforms, np.float64).reshape(B, k + 1)
    j = res["num_accepted"]
    valid = j >= 0
    P, Q = dbg[:, :k], dbg[:, k:2 * k]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(Q > 0, P / Q, np.inf)
    tested = np.arange(k)[None, :] <= np.minimum(j, k - 1)[:, None]
    acc = np.any(tested & (np.abs(u[:, :k] - ratio) < tol), axis=1)
    S, c0, c1 = dbg[:, 2 * k], dbg[:, 2 * k + 1], dbg[:, 2 * k + 2]
    with np.errstate(divide="ignore", invalid="ignore"):
        cdf = (np.abs(u[:, k] - c0 / S) < tol) | (np.abs(u[:, k] - c1 / S) < tol)
    nuc = np.zeros(B, bool)
    if top_p < 1.0:
        near = (np.abs(info[:, :, 2] - top_p) < tol) | (np.abs(info[:, :, 3] - top_p) < tol)
        nuc = np.any(near, axis=1)
    return acc & valid, cdf & valid, nuc & valid


def boundary_flags(res, uniforms, top_p=1.0, tol=1e-5):
    """Sequences within `tol` of any decision boundary (the union of
    boundary_kinds)."""
    acc, cdf, nuc = boundary_kinds(res, uniforms, top_p, tol)
    return acc | cdf | nuc


def verify_tree_sample(target, draft, parents, node_tokens, uniforms, depth, T=1.0, top_p=1.0,
                       top_k=0):
    """Stochastic tree verification (reading R11).  target, draft [B, N, V];
    parents [N]; node_tokens [B, N]; uniforms [B, N] (entry 0: the final
    draw, entry c: node c's test).  Returns dict(tokens [B, D+1],
    num_accepted [B], path [B, D+1], margin [B], errors)."""
    tgt, dt = _logits(target)
    drf, dt2 = _logits(draft)
    B, N, V = tgt.shape
    if dt2 != dt or drf.shape != (B, N, V):
        raise ValueError("draft logits must match target dtype and be [B, N, V]")
    par = np.ascontiguousarray(parents, np.int32)
    tok = np.ascontiguousarray(node_tokens, np.int32).reshape(B, N)
    uni = np.ascontiguousarray(uniforms, np.float32).reshape(B, N)
    W = depth + 1
    out_t = np.zeros((B, W), np.int32)
    out_n = np.zeros(B, np.int32)
    out_p = np.zeros((B, W), np.int32)
    mg = np.zeros(B, np.float64)
    err = _load().oracle_verify_tree_sample(_ptr(tgt), _ptr(drf), dt, _ptr(par), _ptr(tok),
                                            _ptr(uni), B, N, V, int(depth), float(T),
                                            float(top_p), int(top_k), _ptr(out_t), _ptr(out_n),
                                            _ptr(out_p), _ptr(mg))
    if err < 0:
        raise ValueError("oracle_verify_tree_sample rejected its arguments")
    return dict(tokens=out_t, num_accepted=out_n, path=out_p, margin=mg, errors=err)
