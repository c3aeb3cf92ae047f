"""The C ABI library: builds, loads, exports every declared symbol, and
rejects bad arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specsel.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def sd():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import __graft_entry__ as g
    g._load_build_module().build()
    import speculative_decoding_draft_column_gb300 as sd
    return sd


def test_every_declared_symbol_is_exported(sd):
    names = declared_functions()
    assert len(names) >= 12, names
    raw = ctypes.CDLL(sd.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in specsel.h but not exported"
    assert set(names) == set(sd.EXPORTS), "Python binding and header disagree"


def test_host_argument_checks(sd):
    lib = sd.lib
    P = 0x100000          # never dereferenced: every call below fails its checks first
    A = sd.SPEC_ERR_ARG
    assert lib.spec_topk(None, 1, 10, 3, P, P) == A
    assert lib.spec_topk(P, 1, 10, 0, P, P) == A
    assert lib.spec_topk(P, 1, 10, 11, P, P) == A
    assert lib.spec_topk(P, 1, 100, 65, P, P) == A
    assert lib.spec_topk(P, 1, 0, 1, P, P) == A
    assert lib.spec_topk(P, -1, 10, 1, P, P) == A
    assert lib.spec_topk(P + 1, 1, 10, 1, P, P) == A        # logits not 2-byte aligned
    assert lib.spec_topk(P, 1, 10, 1, P, P + 2) == A        # ids not 4-byte aligned
    assert "aligned" in sd.spec_last_error()
    assert lib.spec_topk_mapped(P, 1, 10, 2, None, P, P) == A
    assert lib.spec_verify(P, P, 1, 0, P, P) == A
    assert lib.spec_verify(P, P, 1, 16, P, P) == A
    assert lib.spec_verify(None, P, 1, 7, P, P) == A
    assert lib.spec_verify_v(P, P, 1, 7, 0, P, P) == A
    assert lib.spec_round(P, 1, 10, 3, P, P, P, P, 1, 16, P, P) == A
    assert "gamma" in sd.spec_last_error()
    assert lib.spec_reserve(10, 65, 1, 1) == A
    # empty problems are no-ops that succeed without any CUDA call
    assert lib.spec_topk(None, 0, 10, 3, None, None) == sd.SPEC_OK
    assert lib.spec_verify(None, None, 0, 7, None, None) == sd.SPEC_OK
    assert lib.spec_round(None, 0, 10, 3, None, None, None, None, 0, 7, None, None) == sd.SPEC_OK
    assert sd.spec_last_error() == ""
    assert sd.spec_launch_count() == 0


def test_python_binding_raises(sd):
    with pytest.raises(sd.SpecError) as ei:
        sd.spec_topk(None, 1, 10, 3, None, None)
    assert ei.value.status == sd.SPEC_ERR_ARG


def test_stream_is_thread_local(sd):
    import threading
    sd.lib.spec_set_stream(ctypes.c_void_p(0x1234))
    seen = []
    t = threading.Thread(target=lambda: seen.append(sd.lib.spec_get_stream()))
    t.start(); t.join()
    assert sd.lib.spec_get_stream() == 0x1234 and seen == [None]
    sd.lib.spec_set_stream(None)


def test_kernel_choice(sd):
    assert sd.spec_get_kernel() == sd.SPEC_KERNEL_AUTO
    for which in (sd.SPEC_KERNEL_WARP, sd.SPEC_KERNEL_CTA, sd.SPEC_KERNEL_GROUPMAX, sd.SPEC_KERNEL_AUTO):
        assert sd.lib.spec_set_kernel(which) == sd.SPEC_OK
        assert sd.spec_get_kernel() == which
    for bad in (-1, 4, 99):
        assert sd.lib.spec_set_kernel(bad) == sd.SPEC_ERR_ARG
        assert "unknown kernel" in sd.spec_last_error()
    assert sd.spec_get_kernel() == sd.SPEC_KERNEL_AUTO


def test_counted_round_checks_counters_alignment(sd):
    lib = sd.lib
    P = 0x10000   # never dereferenced: the call fails its argument checks first
    st = lib.spec_round_counted(P, 2, 100, 3, P, P, P, P, 1, 2, P, P, P + 4)
    assert st == sd.SPEC_ERR_ARG and "counters misaligned" in sd.spec_last_error()
    assert sd.COUNTER_WORDS == 3 + 2 * sd.SPEC_MAX_GAMMA


def test_sampled_verify_argument_checks(sd):
    lib = sd.lib
    P = 0x10000   # never dereferenced: every call below fails its checks first
    for T, p, k, msg in [(0.0, 0.95, 20, "temperature"), (-1.0, 0.95, 20, "temperature"),
                         (1.0, 0.0, 20, "top_p"), (1.0, 1.5, 20, "top_p"), (1.0, 0.95, 0, "top_k"),
                         (1.0, 0.95, 65, "top_k"), (1.0, 0.95, 11, "top_k")]:
        st = lib.spec_verify_sampled(P, P, 1, 2, 10, T, p, k, P, P, P)
        assert st == sd.SPEC_ERR_ARG and msg in sd.spec_last_error(), (T, p, k)
    assert lib.spec_verify_sampled(P, P, 1, 2, 100, 1.0, 0.95, 20, None, P, P) == sd.SPEC_ERR_ARG
    assert lib.spec_verify_sampled(P, P, 1, 2, 100, 1.0, 0.95, 20, P + 4, P, P) == sd.SPEC_ERR_ARG
    assert lib.spec_verify_sampled(None, None, 0, 2, 100, 1.0, 0.95, 20, None, None, None) == sd.SPEC_OK


def test_noalloc_limits_checked_per_term_on_host(sd):
    """spec_round_noalloc rejects sizes beyond its fixed scratch on the host,
    each term on its own, so no sum of huge sizes can wrap past the check."""
    lib = sd.lib
    P = 0x100000          # never dereferenced: every call below fails its checks first
    A = sd.SPEC_ERR_ARG
    assert lib.spec_round_noalloc(P, 9000, 1000, 8, P, P, P, P, 1, 7, P, P) == A       # draft columns alone
    assert "8192" in sd.spec_last_error()
    assert lib.spec_round_noalloc(P, 1, 1000, 8, P, P, P, P, 513, 1, P, P) == A        # lanes alone
    assert "512" in sd.spec_last_error()
    assert lib.spec_round_noalloc(P, 8000, 1000, 8, P, P, P, P, 64, 7, P, P) == A      # the sum
    # lanes * (gamma + 1) near 2^63 with V = 1: passes the generic size checks,
    # and cols + lanes * (gamma + 1) would wrap negative
    huge = (2 ** 63 - 1) // 2 - 8
    assert lib.spec_round_noalloc(P, 100, 1, 1, P, P, P, P, huge, 1, P, P) == A
    assert lib.spec_launch_count() == 0


def test_shortlist_head_argument_checks(sd):
    lib = sd.lib
    P = 0x100000          # never dereferenced: every call below fails its checks first
    A = sd.SPEC_ERR_ARG
    assert lib.spec_shortlist_pack(P, P, 24, 128, P, P) == A        # rows not a multiple of 16
    assert lib.spec_shortlist_pack(P, P, 32, 96, P, P) == A         # d not a multiple of 64
    assert lib.spec_shortlist_pack(P, P, 32, 8192, P, P) == A       # d above the staged maximum
    assert lib.spec_shortlist_pack(P, P, 32, 128, P + 8, P) == A    # packed weights not 16-byte aligned
    assert lib.spec_shortlist_logits(P + 2, 1, 128, P, P, 32, P) == A   # hidden not 4-byte aligned
    assert lib.spec_shortlist_topk(P, 1, 128, P, P, 32, P, 33, P, P, P) == A   # k > rows
    assert lib.spec_shortlist_logits(None, 0, 128, P, P, 32, None) == sd.SPEC_OK
    assert lib.spec_launch_count() == 0
