"""Helpers for the GPU parity tests: device copies with guard bands, and the
comparison against the oracle (bit-exact everywhere: ids, bf16 bits, accept
lengths and committed ids)."""
from __future__ import annotations

import numpy as np

import oracle

GUARD = 2048                     # elements of sentinel on each side of an output
SENT16, SENT32 = 0x5A5A, 0x5A5A5A5A


def sd_module():
    import speculative_decoding_draft_column_gb300 as sd
    return sd


def dev_u16(a: np.ndarray, offset: int = 0):
    """uint16 host array -> int16 CUDA tensor, optionally starting `offset`
    elements into a larger allocation (to vary the 16-byte phase)."""
    import torch
    a = np.ascontiguousarray(a, dtype=np.uint16)
    flat = torch.empty(a.size + offset + 8, dtype=torch.int16, device="cuda")
    flat.fill_(0x7F7F)
    v = flat[offset: offset + a.size]
    v.copy_(torch.from_numpy(a.reshape(-1).view(np.int16)))
    return v.view(a.shape)


def dev_i32(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


class Guarded:
    """An output buffer of n elements with sentinel bands on both sides."""

    def __init__(self, n: int, dtype):
        import torch
        self.n = n
        self.dtype = dtype
        self.sent = SENT16 if dtype == torch.int16 else SENT32      # both fit the signed type
        self.buf = torch.full((n + 2 * GUARD,), self.sent, dtype=dtype, device="cuda")
        self.view = self.buf[GUARD: GUARD + n]

    def check_guards(self):
        b = self.buf.cpu().numpy()
        assert np.all(b[:GUARD] == self.sent) and np.all(b[GUARD + self.n:] == self.sent), "guard band overwritten"

    def host(self):
        return self.view.cpu().numpy()


def run_topk(x_host: np.ndarray, k: int, offset: int = 0, id_map: np.ndarray | None = None):
    import torch
    sd = sd_module()
    cols, V = x_host.shape
    x = dev_u16(x_host, offset)
    vals = Guarded(cols * k, torch.int16)
    ids = Guarded(cols * k, torch.int32)
    if id_map is None:
        sd.spec_topk(x, cols, V, k, vals.view, ids.view)
    else:
        sd.spec_topk_mapped(x, cols, V, k, dev_i32(id_map), vals.view, ids.view)
    torch.cuda.synchronize()
    sd.spec_device_status()
    vals.check_guards()
    ids.check_guards()
    return vals.host().view(np.uint16).reshape(cols, k), ids.host().reshape(cols, k)


def run_verify(t_host: np.ndarray, drafts: np.ndarray, offset: int = 0):
    import torch
    sd = sd_module()
    lanes, gamma = drafts.shape
    V = t_host.shape[-1]
    t = dev_u16(t_host, offset)
    acc = Guarded(lanes, torch.int32)
    com = Guarded(lanes * (gamma + 1), torch.int32)
    sd.spec_verify_v(t, dev_i32(drafts), lanes, gamma, V, acc.view, com.view)
    torch.cuda.synchronize()
    sd.spec_device_status()
    acc.check_guards()
    com.check_guards()
    return acc.host(), com.host().reshape(lanes, gamma + 1)


def run_round(x_host, k, t_host, drafts, offset: int = 0):
    import torch
    sd = sd_module()
    cols, V = x_host.shape
    lanes, gamma = drafts.shape
    x = dev_u16(x_host, offset)
    t = dev_u16(t_host, (offset * 3) % 8)
    vals = Guarded(cols * k, torch.int16)
    ids = Guarded(cols * k, torch.int32)
    acc = Guarded(lanes, torch.int32)
    com = Guarded(lanes * (gamma + 1), torch.int32)
    sd.spec_round(x, cols, V, k, vals.view, ids.view, t, dev_i32(drafts), lanes, gamma, acc.view, com.view)
    torch.cuda.synchronize()
    sd.spec_device_status()
    for g in (vals, ids, acc, com):
        g.check_guards()
    return (vals.host().view(np.uint16).reshape(cols, k), ids.host().reshape(cols, k), acc.host(),
            com.host().reshape(lanes, gamma + 1))


def assert_topk_equal(got, want, what=""):
    gv, gi = got
    wv, wi = want
    if not (np.array_equal(gi, wi) and np.array_equal(gv, wv)):
        bad = np.nonzero(np.any(gi != wi, axis=1) | np.any(gv != wv, axis=1))[0]
        c = int(bad[0])
        raise AssertionError(f"{what}: {len(bad)} columns differ; first column {c}:\n"
                             f"  ids  got {gi[c].tolist()}\n       want {wi[c].tolist()}\n"
                             f"  vals got {[hex(v) for v in gv[c]]}\n       want {[hex(v) for v in wv[c]]}")


def assert_verify_equal(got, want, what=""):
    ga, gc = got
    wa, wc = want
    assert np.array_equal(ga, wa), f"{what}: accept lengths differ: got {ga.tolist()} want {wa.tolist()}"
    assert np.array_equal(gc, wc), f"{what}: commit ids differ:\n got {gc.tolist()}\nwant {wc.tolist()}"


def oracle_topk(x, k, id_map=None):
    if id_map is None:
        return oracle.topk(x, k)
    return oracle.topk_mapped(x, k, id_map)


def run_verify_sampled(t_host: np.ndarray, drafts: np.ndarray, temperature: float, top_p: float, top_k: int,
                       uniforms: np.ndarray, offset: int = 0):
    import torch
    sd = sd_module()
    lanes, gamma = drafts.shape
    V = t_host.shape[-1]
    t = dev_u16(t_host, offset)
    u = torch.from_numpy(np.ascontiguousarray(uniforms, dtype=np.float64)).cuda()
    acc = Guarded(lanes, torch.int32)
    com = Guarded(lanes * (gamma + 1), torch.int32)
    sd.spec_verify_sampled(t, dev_i32(drafts), lanes, gamma, V, temperature, top_p, top_k, u, acc.view, com.view)
    torch.cuda.synchronize()
    sd.spec_device_status()
    acc.check_guards()
    com.check_guards()
    return acc.host(), com.host().reshape(lanes, gamma + 1)
