"""ctypes wrapper around the CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm are the only users.  The library in
``speculative_decoding_draft_column_gb300`` never imports this package.

All arrays are numpy; bf16 values travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_NAN, ERR_NOMEM = 0, -1, -2, -3


def build(src: str = _SRC, out: str = _LIB, extra: tuple[str, ...] = ()) -> str:
    """Compile the oracle with gcc (plain C11, no CUDA)."""
    cmd = ["gcc", "-std=c11", "-O2", "-shared", "-fPIC", "-pthread", *extra, src, "-o", out]
    subprocess.run(cmd, check=True)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; returns a ctypes CDLL."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _bind(lib):
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.oracle_topk.argtypes = [p, i64, i64, i32, p, p, ctypes.c_int]
    lib.oracle_topk_mapped.argtypes = [p, i64, i64, i32, p, p, p, ctypes.c_int]
    lib.oracle_argmax.argtypes = [p, i64, i64, p, ctypes.c_int]
    lib.oracle_verify.argtypes = [p, p, i64, i32, i64, p, p, ctypes.c_int]
    for f in (lib.oracle_topk, lib.oracle_topk_mapped, lib.oracle_argmax, lib.oracle_verify):
        f.restype = ctypes.c_int
    return lib


class OracleError(RuntimeError):
    pass


def _check(st: int):
    if st != OK:
        raise OracleError({ERR_ARG: "argument error", ERR_NAN: "NaN in input (outside the contract)",
                           ERR_NOMEM: "out of memory"}.get(st, f"status {st}"))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def topk(logits: np.ndarray, k: int, threads: int | None = None, lib=None):
    """Per-column top-k of a [cols, V] uint16 (bf16) matrix -> (vals u16, ids i32)."""
    lib = lib or load()
    x = np.ascontiguousarray(logits, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    cols, V = x.shape
    vals = np.zeros((cols, k), dtype=np.uint16)
    ids = np.zeros((cols, k), dtype=np.int32)
    _check(lib.oracle_topk(_ptr(x), cols, V, k, _ptr(vals), _ptr(ids), threads or default_threads()))
    return vals, ids


def topk_mapped(logits: np.ndarray, k: int, id_map: np.ndarray, threads: int | None = None, lib=None):
    """Shortlist top-k: ties and output ids are vocabulary ids ``id_map[local]``."""
    lib = lib or load()
    x = np.ascontiguousarray(logits, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    cols, V = x.shape
    m = np.ascontiguousarray(id_map, dtype=np.int32)
    assert m.shape == (V,)
    vals = np.zeros((cols, k), dtype=np.uint16)
    ids = np.zeros((cols, k), dtype=np.int32)
    _check(lib.oracle_topk_mapped(_ptr(x), cols, V, k, _ptr(m), _ptr(vals), _ptr(ids),
                                  threads or default_threads()))
    return vals, ids


def argmax(logits: np.ndarray, threads: int | None = None, lib=None):
    lib = lib or load()
    x = np.ascontiguousarray(logits, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    cols, V = x.shape
    out = np.zeros(cols, dtype=np.int32)
    _check(lib.oracle_argmax(_ptr(x), cols, V, _ptr(out), threads or default_threads()))
    return out


def verify(target: np.ndarray, drafts: np.ndarray, threads: int | None = None, lib=None):
    """Greedy verify: target [lanes*(gamma+1), V], drafts [lanes, gamma]."""
    lib = lib or load()
    d = np.ascontiguousarray(drafts, dtype=np.int32)
    lanes, gamma = d.shape
    t = np.ascontiguousarray(target, dtype=np.uint16).reshape(lanes * (gamma + 1), -1)
    V = t.shape[1]
    acc = np.zeros(lanes, dtype=np.int32)
    com = np.zeros((lanes, gamma + 1), dtype=np.int32)
    _check(lib.oracle_verify(_ptr(t), _ptr(d), lanes, gamma, V, _ptr(acc), _ptr(com),
                             threads or default_threads()))
    return acc, com


def counters(accept_len: np.ndarray, gamma: int) -> dict:
    """The round counters of one verify round ("A drafter inside the
    artifact", Ignis DFlash2 page, section "See it, control it", Metrics):
    per lane one round, gamma drafted tokens and its accept length a of
    accepted tokens; per position i < gamma one drafted token, and one
    accepted token when a > i.  Written out lane by lane, position by
    position (small inputs only)."""
    acc = [int(a) for a in np.asarray(accept_len).reshape(-1)]
    out = {"rounds": 0, "drafted_tokens": 0, "accepted_tokens": 0,
           "position_drafted": [0] * gamma, "position_accepted": [0] * gamma}
    for a in acc:
        if not 0 <= a <= gamma:
            raise ValueError(f"accept length {a} outside [0, {gamma}]")
        out["rounds"] += 1
        out["drafted_tokens"] += gamma
        out["accepted_tokens"] += a
        for i in range(gamma):
            out["position_drafted"][i] += 1
            if a > i:
                out["position_accepted"][i] += 1
    return out


def sampled_column(values: np.ndarray, ids: np.ndarray, temperature: float, top_p: float):
    """The target's sampling distribution over one column's top-k set
    ("A drafter inside the artifact", Ignis DFlash2 page, "The numbers":
    sampled acceptance at T, top_p, top_k).  values: the top-k bf16 bits,
    best first (ties by smaller id), ids: their token ids.  Steps, each in
    float64 and in this order: z_t = v_t / T; e_t = exp(z_t - z_0); S = sum of
    e_t in list order; p_t = e_t / S; the nucleus is the shortest prefix whose
    running sum c_t (list order) reaches top_p; q_t = p_t / c_last on it.
    Returns (kept ids, q)."""
    vals = np.asarray(values, dtype=np.uint16).astype(np.uint32) << 16
    x = vals.view(np.float32).astype(np.float64)
    z = [float(xi) / temperature for xi in x]
    e = [np.exp(zi - z[0]) for zi in z]
    S = 0.0
    for ei in e:
        S += ei
    p = [ei / S for ei in e]
    c, last = 0.0, len(p) - 1
    for t, pt in enumerate(p):
        c += pt
        if c >= top_p:
            last = t
            break
    kept = [int(i) for i in ids[:last + 1]]
    q = [p[t] / c for t in range(last + 1)]
    return kept, q


def sampled_decision(kept, q, draft: int | None, u: float, u2: float):
    """One position of sampled verify with a one-hot draft: accept the draft
    when u < q(draft) (q = 0 outside the nucleus); otherwise (or with no
    draft, the bonus position) draw from q with the draft's mass removed:
    the first kept token (list order, the draft skipped) whose running weight
    exceeds u2 times the total weight.  Returns (accepted, token, margin):
    token is the draft when accepted, else the draw; margin is the smallest
    distance of u or u2 (scaled) to a decision boundary."""
    qd = 0.0
    if draft is not None:
        for t, tok in enumerate(kept):
            if tok == draft:
                qd = q[t]
        if u < qd:
            return True, int(draft), abs(u - qd)
    margin = abs(u - qd) if draft is not None else float("inf")
    W = 0.0
    for t, tok in enumerate(kept):
        if draft is None or tok != draft:
            W += q[t]
    target = u2 * W
    run, pick = 0.0, None
    for t, tok in enumerate(kept):
        if draft is not None and tok == draft:
            continue
        prev = run
        run += q[t]
        if pick is None and run > target:
            pick = tok
            margin = min(margin, abs(target - prev), abs(run - target))
    if pick is None:   # rounding left the target at the very end: the last kept token
        pick = [tok for tok in kept if draft is None or tok != draft][-1]
        margin = 0.0
    return False, int(pick), margin


def sampled_verify(target: np.ndarray, drafts: np.ndarray, temperature: float, top_p: float, top_k: int,
                   uniforms: np.ndarray, threads: int | None = None):
    """Sampled verify with one-hot drafts (speculative sampling): target
    [lanes*(gamma+1), V] bf16 bits, drafts [lanes, gamma], uniforms
    [lanes, gamma+1, 2] in [0, 1).  Position j < gamma accepts draft j with
    probability q_j(draft j); the first rejection commits a draw from q_j
    without the draft, and a lane that accepts all gamma drafts commits a
    bonus draw from q_gamma.  Returns (accept_len, commit_ids, min margin)."""
    d = np.ascontiguousarray(drafts, dtype=np.int32)
    lanes, gamma = d.shape
    t = np.ascontiguousarray(target, dtype=np.uint16).reshape(lanes * (gamma + 1), -1)
    u = np.asarray(uniforms, dtype=np.float64).reshape(lanes, gamma + 1, 2)
    vals, ids = topk(t, top_k, threads=threads)
    acc = np.zeros(lanes, dtype=np.int32)
    com = np.full((lanes, gamma + 1), -1, dtype=np.int32)
    margin = float("inf")
    for ln in range(lanes):
        a = gamma
        for j in range(gamma + 1):
            kept, q = sampled_column(vals[ln * (gamma + 1) + j], ids[ln * (gamma + 1) + j], temperature, top_p)
            draft = int(d[ln, j]) if j < gamma else None
            ok, tok, m = sampled_decision(kept, q, draft, float(u[ln, j, 0]), float(u[ln, j, 1]))
            margin = min(margin, m)
            com[ln, j] = tok
            if not ok:
                a = j
                break
        acc[ln] = a
    return acc, com, margin
