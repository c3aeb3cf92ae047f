"""The Python binding's buffer checks (no GPU): a tensor argument must be a
contiguous CUDA tensor large enough for the call, else SpecError(SPEC_ERR_ARG)
is raised before anything reaches the library.  Device tensors are stood in
for by objects with a tensor's attributes; calls that pass the checks reach
the C library, which (without a GPU) fails with SPEC_ERR_CUDA at its first
CUDA call -- those tests are skipped where a GPU is present, so that their
stand-in pointers never reach a kernel."""
import os
import shutil
from types import SimpleNamespace

import numpy as np
import pytest


@pytest.fixture(scope="module")
def sd():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import __graft_entry__ as g
    g._load_build_module().build()
    import speculative_decoding_draft_column_gb300 as m
    return m


class Dev:
    """A stand-in CUDA tensor of n elements of `elem` bytes."""

    def __init__(self, n, elem=2, contiguous=True, ptr=0x100000):
        self.n, self.elem, self.contig, self.ptr = n, elem, contiguous, ptr
        self.is_cuda = True
        self.device = SimpleNamespace(index=0, type="cuda")

    def is_contiguous(self):
        return self.contig

    def numel(self):
        return self.n

    def element_size(self):
        return self.elem

    def data_ptr(self):
        return self.ptr


def _no_gpu():
    import torch
    return not torch.cuda.is_available()


def _rejected(sd, fn, *args, match):
    with pytest.raises(sd.SpecError) as ei:
        fn(*args)
    assert ei.value.status == sd.SPEC_ERR_ARG and match in str(ei.value), str(ei.value)


def _reaches_library(sd, fn, *args):
    with pytest.raises(sd.SpecError) as ei:
        fn(*args)
    assert ei.value.status == sd.SPEC_ERR_CUDA, str(ei.value)


def test_host_tensor_for_device_argument(sd):
    import torch
    x = torch.zeros((2, 10), dtype=torch.int16)
    _rejected(sd, sd.spec_topk, x, 2, 10, 3, Dev(6), Dev(6, 4), match="logits: need a CUDA tensor")


def test_non_contiguous_and_short_buffers(sd):
    cols, V, k = 3, 100, 8
    _rejected(sd, sd.spec_topk, Dev(cols * V, contiguous=False), cols, V, k, Dev(cols * k), Dev(cols * k, 4),
              match="logits: tensor must be contiguous")
    _rejected(sd, sd.spec_topk, Dev(cols * V - 1), cols, V, k, Dev(cols * k), Dev(cols * k, 4),
              match="logits: 598 bytes, the call needs 600")
    _rejected(sd, sd.spec_topk, Dev(cols * V), cols, V, k, Dev(cols * k), Dev(cols * k - 1, 4),
              match="out_ids")
    _rejected(sd, sd.spec_topk_mapped, Dev(cols * V), cols, V, k, Dev(V - 1, 4), Dev(cols * k), Dev(cols * k, 4),
              match="id_map")
    lanes, gamma = 2, 3
    t, d = Dev(lanes * (gamma + 1) * V), Dev(lanes * gamma, 4)
    a, c = Dev(lanes, 4), Dev(lanes * (gamma + 1), 4)
    _rejected(sd, sd.spec_verify_v, t, Dev(lanes * gamma - 1, 4), lanes, gamma, V, a, c, match="drafts")
    _rejected(sd, sd.spec_verify_v, t, d, lanes, gamma, V, a, Dev(lanes * gamma, 4), match="out_commit_ids")
    _rejected(sd, sd.spec_verify, t, d, lanes, gamma, a, c, match="target_logits")   # V is the vocabulary
    _rejected(sd, sd.spec_verify_sampled, t, d, lanes, gamma, V, 1.0, 0.95, 20, Dev(lanes * (gamma + 1) * 2 - 1, 8),
              a, c, match="uniforms")
    _rejected(sd, sd.spec_round_counted, Dev(cols * V), cols, V, k, Dev(cols * k), Dev(cols * k, 4), t, d, lanes,
              gamma, a, c, Dev(sd.COUNTER_WORDS - 1, 8), match="counters")


def test_host_buffers_checked(sd):
    cols, V, k, lanes, gamma = 2, 50, 4, 1, 2
    x = np.zeros((cols, V), dtype=np.uint16)
    t = np.zeros((lanes * (gamma + 1), V), dtype=np.uint16)
    d = np.zeros((lanes, gamma), dtype=np.int32)
    v, i = np.zeros((cols, k), dtype=np.uint16), np.zeros((cols, k), dtype=np.int32)
    a, c = np.zeros(lanes, dtype=np.int32), np.zeros((lanes, gamma + 1), dtype=np.int32)
    _rejected(sd, sd.spec_round_host, x[:, ::2], cols, V, k, v, i, t, d, lanes, gamma, a, c,
              match="C-contiguous")
    _rejected(sd, sd.spec_round_host, x, cols, V, k, v[:1], i, t, d, lanes, gamma, a, c, match="out_vals")
    _rejected(sd, sd.spec_round_host, x, cols, V, k, v, i, t[:2], d, lanes, gamma, a, c, match="target_logits")
    _rejected(sd, sd.spec_round_host, x, cols, V, k, v, i, t, d, lanes, gamma, a, Dev(3, 4), match="host array")


def test_empty_calls_and_raw_pointers_pass_unchecked(sd):
    # zero columns / lanes need no buffers; raw integer pointers are not checked
    sd.spec_topk(Dev(0), 0, 10, 3, Dev(0), Dev(0, 4))
    sd.spec_verify_v(None, None, 0, 2, 10, None, None)
    with pytest.raises(sd.SpecError) as ei:
        sd.spec_topk(None, 1, 10, 3, None, None)           # the C check
    assert ei.value.status == sd.SPEC_ERR_ARG and "null pointer" in str(ei.value)


@pytest.mark.skipif(not _no_gpu(), reason="stand-in pointers must not reach a kernel")
def test_exact_sizes_reach_the_library(sd):
    cols, V, k, lanes, gamma = 3, 100, 8, 2, 3
    x, v, i = Dev(cols * V), Dev(cols * k), Dev(cols * k, 4)
    t, d = Dev(lanes * (gamma + 1) * V), Dev(lanes * gamma, 4)
    a, c = Dev(lanes, 4), Dev(lanes * (gamma + 1), 4)
    u = Dev(lanes * (gamma + 1) * 2, 8)
    _reaches_library(sd, sd.spec_topk, x, cols, V, k, v, i)
    _reaches_library(sd, sd.spec_topk_mapped, x, cols, V, k, Dev(V, 4), v, i)
    _reaches_library(sd, sd.spec_verify_v, t, d, lanes, gamma, V, a, c)
    _reaches_library(sd, sd.spec_verify, Dev(lanes * (gamma + 1) * sd.SPEC_VOCAB), d, lanes, gamma, a, c)
    _reaches_library(sd, sd.spec_round, x, cols, V, k, v, i, t, d, lanes, gamma, a, c)
    _reaches_library(sd, sd.spec_round_noalloc, x, cols, V, k, v, i, t, d, lanes, gamma, a, c)
    _reaches_library(sd, sd.spec_round_counted, x, cols, V, k, v, i, t, d, lanes, gamma, a, c,
                     Dev(sd.COUNTER_WORDS, 8))
    _reaches_library(sd, sd.spec_verify_sampled, t, d, lanes, gamma, V, 1.0, 0.95, 20, u, a, c)
    _reaches_library(sd, sd.spec_round_sampled, x, cols, V, k, v, i, t, d, lanes, gamma, 1.0, 0.95, 20, u, a, c)
    hx = np.zeros((cols, V), dtype=np.uint16)
    ht = np.zeros((lanes * (gamma + 1), V), dtype=np.uint16)
    hd = np.zeros((lanes, gamma), dtype=np.int32)
    hv, hi = np.zeros((cols, k), dtype=np.uint16), np.zeros((cols, k), dtype=np.int32)
    ha, hc = np.zeros(lanes, dtype=np.int32), np.zeros((lanes, gamma + 1), dtype=np.int32)
    _reaches_library(sd, sd.spec_round_host, hx, cols, V, k, hv, hi, ht, hd, lanes, gamma, ha, hc)
