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
