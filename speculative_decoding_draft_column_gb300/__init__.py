"""Python binding of libspecsel (the C ABI declared in ``include/specsel.h``).

Argument marshalling only: every function below with a C name forwards its
arguments to the C entry point of the same name -- device tensors become
device pointers, and the call is enqueued on PyTorch's current CUDA stream.
All selection work runs in the CUDA kernels of ``csrc/specsel.cu``; there
is no CPU or PyTorch fallback.  If the shared library has not been built
(``__graft_entry__.build()``), importing this package raises ImportError.

Tensor conventions: bf16 logits may be ``torch.bfloat16`` or a 16-bit
integer view of the same bits; ids and lengths are ``torch.int32``.  A
tensor argument must be contiguous, on the current CUDA device (host memory
for ``spec_round_host``) and hold at least what the call reads or writes;
otherwise ``SpecError`` (``SPEC_ERR_ARG``) is raised before the library is
called.  Raw integer pointers are passed on unchecked, as in the C ABI.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "SPEC_OK", "SPEC_ERR_ARG", "SPEC_ERR_ALLOC", "SPEC_ERR_CUDA", "SPEC_VOCAB", "SPEC_MAX_K",
    "SPEC_MAX_GAMMA", "SpecError", "LIB_PATH", "lib",
    "spec_topk", "spec_topk_mapped", "spec_verify", "spec_verify_v", "spec_round", "spec_round_host",
    "spec_round_noalloc", "spec_round_counted", "spec_verify_sampled", "spec_round_sampled", "new_counters", "read_counters", "COUNTER_WORDS",
    "spec_set_kernel", "spec_get_kernel", "spec_last_kernel", "SPEC_KERNEL_AUTO", "SPEC_KERNEL_WARP", "SPEC_KERNEL_CTA",
    "SPEC_KERNEL_GROUPMAX",
    "spec_set_stream", "spec_get_stream", "spec_reserve", "spec_release", "spec_last_error",
    "spec_launch_count", "spec_device_status", "topk", "topk_mapped", "verify", "round_step", "EXPORTS",
    "spec_shortlist_pack", "spec_shortlist_logits", "spec_shortlist_topk",
]

SPEC_OK, SPEC_ERR_ARG, SPEC_ERR_ALLOC, SPEC_ERR_CUDA = 0, -1, -2, -3
SPEC_VOCAB, SPEC_MAX_K, SPEC_MAX_GAMMA = 248_046, 64, 15
SPEC_KERNEL_AUTO, SPEC_KERNEL_WARP, SPEC_KERNEL_CTA, SPEC_KERNEL_GROUPMAX = 0, 1, 2, 3
LIB_PATH = _build.LIB

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                      "(the selection kernels have no CPU fallback)")

lib = ctypes.CDLL(LIB_PATH)

_p, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
_SIGS = {
    "spec_topk": [_p, _i64, _i64, _i32, _p, _p],
    "spec_topk_mapped": [_p, _i64, _i64, _i32, _p, _p, _p],
    "spec_verify": [_p, _p, _i64, _i32, _p, _p],
    "spec_verify_v": [_p, _p, _i64, _i32, _i64, _p, _p],
    "spec_round": [_p, _i64, _i64, _i32, _p, _p, _p, _p, _i64, _i32, _p, _p],
    "spec_round_host": [_p, _i64, _i64, _i32, _p, _p, _p, _p, _i64, _i32, _p, _p],
    "spec_round_noalloc": [_p, _i64, _i64, _i32, _p, _p, _p, _p, _i64, _i32, _p, _p],
    "spec_round_counted": [_p, _i64, _i64, _i32, _p, _p, _p, _p, _i64, _i32, _p, _p, _p],
    "spec_verify_sampled": [_p, _p, _i64, _i32, _i64, ctypes.c_double, ctypes.c_double, _i32, _p, _p, _p],
    "spec_round_sampled": [_p, _i64, _i64, _i32, _p, _p, _p, _p, _i64, _i32, ctypes.c_double, ctypes.c_double, _i32,
                           _p, _p, _p],
    "spec_set_kernel": [_i32],
    "spec_get_kernel": [],
    "spec_last_kernel": [],
    "spec_set_stream": [_p],
    "spec_get_stream": [],
    "spec_reserve": [_i64, _i32, _i64, _i32],
    "spec_release": [],
    "spec_last_error": [],
    "spec_launch_count": [],
    "spec_device_status": [],
    "spec_selftest_wait_timeout": [_i64, _p],
    "spec_shortlist_pack": [_p, _p, _i64, _i64, _p, _p],
    "spec_shortlist_logits": [_p, _i64, _i64, _p, _p, _i64, _p],
    "spec_shortlist_topk": [_p, _i64, _i64, _p, _p, _i64, _p, _i32, _p, _p, _p],
}
EXPORTS = tuple(_SIGS)
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
lib.spec_get_stream.restype = ctypes.c_void_p
lib.spec_last_error.restype = ctypes.c_char_p
lib.spec_launch_count.restype = ctypes.c_int64


class SpecError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"status {status}: {message}")
        self.status = status


def _check(status: int) -> None:
    if status != SPEC_OK:
        raise SpecError(status, lib.spec_last_error().decode(errors="replace"))


def _ptr(x):
    """Device tensor -> pointer; None -> NULL; int -> itself."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _n(x) -> int:
    """A count as a Python int, negatives as 0 (the C checks reject them)."""
    try:
        return max(0, int(x))
    except (TypeError, ValueError):
        return 0


def _dev(x, count, elem_bytes: int, name: str):
    """Pointer of a device buffer that must hold `count` elements of
    `elem_bytes` bytes.  A tensor must be a contiguous CUDA tensor on the
    current device and large enough; otherwise SpecError(SPEC_ERR_ARG) is
    raised before anything is enqueued (a wrong buffer would make a kernel
    read or write outside it).  None and raw integer pointers are passed on
    unchecked, like the C ABI."""
    if x is None or isinstance(x, int):
        return x
    if not (getattr(x, "is_cuda", False) and hasattr(x, "data_ptr")):
        raise SpecError(SPEC_ERR_ARG, f"{name}: need a CUDA tensor (or a raw device pointer)")
    import torch
    if torch.cuda.is_available() and x.device.index != torch.cuda.current_device():
        raise SpecError(SPEC_ERR_ARG, f"{name}: tensor on {x.device}, the current device is "
                                      f"cuda:{torch.cuda.current_device()}")
    if not x.is_contiguous():
        raise SpecError(SPEC_ERR_ARG, f"{name}: tensor must be contiguous")
    need, have = _n(count) * elem_bytes, x.numel() * x.element_size()
    if have < need:
        raise SpecError(SPEC_ERR_ARG, f"{name}: {have} bytes, the call needs {need}")
    return x.data_ptr()


def _host(x, count, elem_bytes: int, name: str):
    """Pointer of a host buffer (numpy array or CPU tensor) of `count`
    elements, checked like `_dev`."""
    if x is None or isinstance(x, int):
        return x
    if hasattr(x, "ctypes") and hasattr(x, "flags"):           # numpy
        if not x.flags.c_contiguous:
            raise SpecError(SPEC_ERR_ARG, f"{name}: array must be C-contiguous")
        have, ptr = x.nbytes, x.ctypes.data
    else:
        if getattr(x, "is_cuda", True) or not hasattr(x, "data_ptr"):
            raise SpecError(SPEC_ERR_ARG, f"{name}: need a host array or CPU tensor")
        if not x.is_contiguous():
            raise SpecError(SPEC_ERR_ARG, f"{name}: tensor must be contiguous")
        have, ptr = x.numel() * x.element_size(), x.data_ptr()
    need = _n(count) * elem_bytes
    if have < need:
        raise SpecError(SPEC_ERR_ARG, f"{name}: {have} bytes, the call needs {need}")
    return ptr


def _topk_bufs(check, logits, cols, V, k, out_vals, out_ids, id_map=None):
    c = _n(cols)
    return (check(logits, c * _n(V), 2, "logits"), check(out_vals, c * _n(k), 2, "out_vals"),
            check(out_ids, c * _n(k), 4, "out_ids"), check(id_map, _n(V) if c else 0, 4, "id_map"))


def _verify_bufs(check, target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids):
    ln, g = _n(lanes), _n(gamma)
    return (check(target_logits, ln * (g + 1) * _n(V), 2, "target_logits"), check(drafts, ln * g, 4, "drafts"),
            check(out_accept_len, ln, 4, "out_accept_len"), check(out_commit_ids, ln * (g + 1), 4, "out_commit_ids"))


def _use_torch_stream():
    import torch
    if torch.cuda.is_available():
        lib.spec_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# ---- same-name wrappers of the C entry points ------------------------------

def spec_topk(logits, cols, V, k, out_vals, out_ids):
    x, v, i, _ = _topk_bufs(_dev, logits, cols, V, k, out_vals, out_ids)
    _use_torch_stream()
    _check(lib.spec_topk(x, cols, V, k, v, i))


def spec_topk_mapped(logits, cols, V, k, id_map, out_vals, out_ids):
    x, v, i, m = _topk_bufs(_dev, logits, cols, V, k, out_vals, out_ids, id_map)
    _use_torch_stream()
    _check(lib.spec_topk_mapped(x, cols, V, k, m, v, i))


def spec_verify(target_logits, drafts, lanes, gamma, out_accept_len, out_commit_ids):
    t, d, a, c = _verify_bufs(_dev, target_logits, drafts, lanes, gamma, SPEC_VOCAB, out_accept_len, out_commit_ids)
    _use_torch_stream()
    _check(lib.spec_verify(t, d, lanes, gamma, a, c))


def spec_verify_v(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids):
    t, d, a, c = _verify_bufs(_dev, target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids)
    _use_torch_stream()
    _check(lib.spec_verify_v(t, d, lanes, gamma, V, a, c))


def spec_round(draft_logits, cols, V, k, out_vals, out_ids, target_logits, drafts, lanes, gamma,
               out_accept_len, out_commit_ids):
    x, v, i, _ = _topk_bufs(_dev, draft_logits, cols, V, k, out_vals, out_ids)
    t, d, a, c = _verify_bufs(_dev, target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids)
    _use_torch_stream()
    _check(lib.spec_round(x, cols, V, k, v, i, t, d, lanes, gamma, a, c))


def spec_round_noalloc(draft_logits, cols, V, k, out_vals, out_ids, target_logits, drafts, lanes, gamma,
                       out_accept_len, out_commit_ids):
    """spec_round with its scratch in a fixed device array: allocates nothing
    (for callers whose device memory all comes from their own pool)."""
    x, v, i, _ = _topk_bufs(_dev, draft_logits, cols, V, k, out_vals, out_ids)
    t, d, a, c = _verify_bufs(_dev, target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids)
    _use_torch_stream()
    _check(lib.spec_round_noalloc(x, cols, V, k, v, i, t, d, lanes, gamma, a, c))


def spec_verify_sampled(target_logits, drafts, lanes, gamma, V, temperature, top_p, top_k, uniforms,
                        out_accept_len, out_commit_ids):
    """Sampled verify with one-hot drafts; ``uniforms`` a float64 CUDA tensor
    [lanes, gamma+1, 2] of numbers in [0, 1)."""
    t, d, a, c = _verify_bufs(_dev, target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids)
    u = _dev(uniforms, _n(lanes) * (_n(gamma) + 1) * 2, 8, "uniforms")
    _use_torch_stream()
    _check(lib.spec_verify_sampled(t, d, lanes, gamma, V, float(temperature), float(top_p), top_k, u, a, c))


def spec_round_sampled(draft_logits, cols, V, k, out_vals, out_ids, target_logits, drafts, lanes, gamma,
                       temperature, top_p, top_k, uniforms, out_accept_len, out_commit_ids):
    """spec_round with sampled verify, one launch."""
    x, v, i, _ = _topk_bufs(_dev, draft_logits, cols, V, k, out_vals, out_ids)
    t, d, a, c = _verify_bufs(_dev, target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids)
    u = _dev(uniforms, _n(lanes) * (_n(gamma) + 1) * 2, 8, "uniforms")
    _use_torch_stream()
    _check(lib.spec_round_sampled(x, cols, V, k, v, i, t, d, lanes, gamma, float(temperature), float(top_p),
                                  top_k, u, a, c))


COUNTER_WORDS = 3 + 2 * SPEC_MAX_GAMMA   # uint64 words of a spec_counters block


def spec_round_counted(draft_logits, cols, V, k, out_vals, out_ids, target_logits, drafts, lanes, gamma,
                       out_accept_len, out_commit_ids, counters):
    """spec_round that also adds the round to ``counters`` (an int64 CUDA
    tensor of COUNTER_WORDS, see ``new_counters``; None: no counting)."""
    x, v, i, _ = _topk_bufs(_dev, draft_logits, cols, V, k, out_vals, out_ids)
    t, d, a, c = _verify_bufs(_dev, target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids)
    n = _dev(counters, COUNTER_WORDS, 8, "counters")
    _use_torch_stream()
    _check(lib.spec_round_counted(x, cols, V, k, v, i, t, d, lanes, gamma, a, c, n))


def new_counters(device="cuda"):
    """A zeroed spec_counters block on the device (int64 tensor)."""
    import torch
    return torch.zeros(COUNTER_WORDS, dtype=torch.int64, device=device)


def read_counters(counters) -> dict:
    """The block as a dict: rounds, drafted_tokens, accepted_tokens,
    position_drafted[15], position_accepted[15]."""
    v = [int(x) for x in counters.cpu().tolist()]
    g = SPEC_MAX_GAMMA
    return {"rounds": v[0], "drafted_tokens": v[1], "accepted_tokens": v[2],
            "position_drafted": v[3:3 + g], "position_accepted": v[3 + g:3 + 2 * g]}


def spec_round_host(draft_logits, cols, V, k, out_vals, out_ids, target_logits, drafts, lanes, gamma,
                    out_accept_len, out_commit_ids):
    """Host buffers (CPU tensors, ideally pinned, or numpy arrays) in and out."""
    x, v, i, _ = _topk_bufs(_host, draft_logits, cols, V, k, out_vals, out_ids)
    t, d, a, c = _verify_bufs(_host, target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids)
    _use_torch_stream()
    _check(lib.spec_round_host(x, cols, V, k, v, i, t, d, lanes, gamma, a, c))


def spec_shortlist_pack(weights, scales, rows, d, wpack, spack):
    """Reorder a Q4 head (uint8 [rows, d/2], fp16 bits [rows, d/64]) into the
    streamed layout (buffers of the same sizes)."""
    r, dd = _n(rows), _n(d)
    w = _dev(weights, r * (dd // 2), 1, "weights")
    sc = _dev(scales, r * (dd // 64), 2, "scales")
    wp = _dev(wpack, r * (dd // 2), 1, "wpack")
    sp = _dev(spack, r * (dd // 64), 2, "spack")
    _use_torch_stream()
    _check(lib.spec_shortlist_pack(w, sc, rows, d, wp, sp))


def _head_bufs(hidden, cols, d, wpack, spack, rows):
    c, r, dd = _n(cols), _n(rows), _n(d)
    return (_dev(hidden, c * dd, 2, "hidden"), _dev(wpack, r * (dd // 2), 1, "wpack"),
            _dev(spack, r * (dd // 64), 2, "spack"))


def spec_shortlist_logits(hidden, cols, d, wpack, spack, rows, out_logits):
    h, wp, sp = _head_bufs(hidden, cols, d, wpack, spack, rows)
    lg = _dev(out_logits, _n(cols) * _n(rows), 2, "out_logits")
    _use_torch_stream()
    _check(lib.spec_shortlist_logits(h, cols, d, wp, sp, rows, lg))


def spec_shortlist_topk(hidden, cols, d, wpack, spack, rows, id_map, k, logits, out_vals, out_ids):
    h, wp, sp = _head_bufs(hidden, cols, d, wpack, spack, rows)
    lg = _dev(logits, _n(cols) * _n(rows), 2, "logits")
    m = _dev(id_map, _n(rows), 4, "id_map")
    v = _dev(out_vals, _n(cols) * _n(k), 2, "out_vals")
    i = _dev(out_ids, _n(cols) * _n(k), 4, "out_ids")
    _use_torch_stream()
    _check(lib.spec_shortlist_topk(h, cols, d, wp, sp, rows, m, k, lg, v, i))


def spec_set_kernel(which: int):
    """Choose the streaming kernel: SPEC_KERNEL_AUTO (default), _WARP, _CTA or _GROUPMAX."""
    _check(lib.spec_set_kernel(which))


def spec_get_kernel() -> int:
    return int(lib.spec_get_kernel())


def spec_last_kernel() -> int:
    """The kernel (SPEC_KERNEL_WARP, _CTA or _GROUPMAX) of this thread's last round launch."""
    return int(lib.spec_last_kernel())


def spec_set_stream(stream):
    """``stream``: a torch.cuda.Stream, a raw cudaStream_t (int) or None."""
    h = getattr(stream, "cuda_stream", stream)
    _check(lib.spec_set_stream(None if h is None else ctypes.c_void_p(h)))


def spec_get_stream():
    return lib.spec_get_stream()


def spec_reserve(max_cols, max_k, max_lanes, max_gamma):
    _check(lib.spec_reserve(max_cols, max_k, max_lanes, max_gamma))


def spec_release():
    _check(lib.spec_release())


def spec_last_error() -> str:
    return lib.spec_last_error().decode(errors="replace")


def spec_launch_count() -> int:
    return int(lib.spec_launch_count())


def spec_device_status():
    """Raise SpecError if a kernel gave up a bounded wait since the last check."""
    _check(lib.spec_device_status())


# ---- allocating conveniences (outputs created with torch, work in the kernels)

def _check_logits(x, name):
    import torch
    if not x.is_cuda or x.dim() != 2 or not x.is_contiguous() or x.element_size() != 2:
        raise ValueError(f"{name}: need a contiguous 2-D CUDA tensor of 16-bit elements")
    if x.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise ValueError(f"{name}: dtype {x.dtype} is not bf16 bits")


def topk(logits, k: int):
    """(vals bf16 [cols,k], ids int32 [cols,k]) for a [cols, V] CUDA tensor."""
    import torch
    _check_logits(logits, "logits")
    cols, V = logits.shape
    vals = torch.empty((cols, k), dtype=logits.dtype, device=logits.device)
    ids = torch.empty((cols, k), dtype=torch.int32, device=logits.device)
    spec_topk(logits, cols, V, k, vals, ids)
    return vals, ids


def topk_mapped(logits, k: int, id_map):
    import torch
    _check_logits(logits, "logits")
    cols, V = logits.shape
    if id_map.dtype != torch.int32 or id_map.numel() != V or not id_map.is_cuda:
        raise ValueError("id_map: need an int32 CUDA tensor with V entries")
    vals = torch.empty((cols, k), dtype=logits.dtype, device=logits.device)
    ids = torch.empty((cols, k), dtype=torch.int32, device=logits.device)
    spec_topk_mapped(logits, cols, V, k, id_map, vals, ids)
    return vals, ids


def verify(target_logits, drafts):
    """target [lanes*(gamma+1), V], drafts int32 [lanes, gamma] -> (accept_len, commit_ids)."""
    import torch
    _check_logits(target_logits, "target_logits")
    lanes, gamma = drafts.shape
    V = target_logits.shape[1]
    if target_logits.shape[0] != lanes * (gamma + 1) or drafts.dtype != torch.int32 or not drafts.is_contiguous():
        raise ValueError("shape mismatch between target_logits and drafts")
    acc = torch.empty(lanes, dtype=torch.int32, device=drafts.device)
    com = torch.empty((lanes, gamma + 1), dtype=torch.int32, device=drafts.device)
    spec_verify_v(target_logits, drafts, lanes, gamma, V, acc, com)
    return acc, com


def round_step(draft_logits, k: int, target_logits, drafts):
    """One fused launch: (vals, ids, accept_len, commit_ids)."""
    import torch
    _check_logits(draft_logits, "draft_logits")
    _check_logits(target_logits, "target_logits")
    cols, V = draft_logits.shape
    lanes, gamma = drafts.shape
    if target_logits.shape != (lanes * (gamma + 1), V):
        raise ValueError("target_logits must be [lanes*(gamma+1), V] with the drafts' V")
    dev = draft_logits.device
    vals = torch.empty((cols, k), dtype=draft_logits.dtype, device=dev)
    ids = torch.empty((cols, k), dtype=torch.int32, device=dev)
    acc = torch.empty(lanes, dtype=torch.int32, device=dev)
    com = torch.empty((lanes, gamma + 1), dtype=torch.int32, device=dev)
    spec_round(draft_logits, cols, V, k, vals, ids, target_logits, drafts, lanes, gamma, acc, com)
    return vals, ids, acc, com
