"""CPU checks of the C ABI: the library loads, exports every entry point the
header declares, and rejects bad arguments on the host before any launch
(these calls never reach the GPU, so they run without one)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "yoco.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"YOCO_API\s+[\w\s\*]+?\b(yoco_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def Y():
    import gated_retention_shared_gb300 as Y
    return Y


def test_header_declares_the_five_calls():
    syms = declared_symbols()
    for name in ("yoco_gret_prefill_chunkwise", "yoco_gret_decode_step", "yoco_shared_kv_project_append",
                 "yoco_cross_attn_prefill", "yoco_cross_attn_decode"):
        assert name in syms


def test_library_exports_every_declared_symbol(Y):
    lib = ctypes.CDLL(Y.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(Y.EXPORTED)


def test_status_strings_and_version(Y):
    assert Y.lib.yoco_version() == 100
    for s in range(7):
        assert Y.lib.yoco_status_string(s)
    assert Y.lib.yoco_status_string(99) == b"unknown status"


FAKE = ctypes.c_void_p(0x1000)  # 16-byte aligned non-null; never dereferenced: every call below fails validation


def _prefill(Y, B=1, N=8, H=1, dk=64, dv=64, chunk=0, in_dt=1, out_dt=1, tau=16.0, state=FAKE):
    return Y.lib.yoco_gret_prefill_chunkwise(FAKE, FAKE, FAKE, FAKE, tau, FAKE, state, B, N, H, dk, dv, chunk,
                                             in_dt, out_dt, None, 0, None)


def test_gret_prefill_rejects_bad_arguments(Y):
    assert _prefill(Y, dk=96, dv=96) == Y.YOCO_ERR_UNSUPPORTED
    assert _prefill(Y, dk=64, dv=128) == Y.YOCO_ERR_UNSUPPORTED
    assert _prefill(Y, in_dt=0, out_dt=1) == Y.YOCO_ERR_UNSUPPORTED
    assert _prefill(Y, in_dt=7, out_dt=7) == Y.YOCO_ERR_INVALID_ARG
    assert _prefill(Y, B=0) == Y.YOCO_ERR_INVALID_ARG
    assert _prefill(Y, N=-1) == Y.YOCO_ERR_INVALID_ARG
    assert _prefill(Y, tau=0.0) == Y.YOCO_ERR_INVALID_ARG
    assert _prefill(Y, tau=float("nan")) == Y.YOCO_ERR_INVALID_ARG
    assert _prefill(Y, chunk=48) == Y.YOCO_ERR_UNSUPPORTED
    assert _prefill(Y, state=None) == Y.YOCO_ERR_INVALID_ARG
    assert b"state" in Y.lib.yoco_last_error()
    # N = 0 is a no-op that touches nothing
    assert _prefill(Y, N=0) == Y.YOCO_OK


def test_gret_prefill_workspace_is_checked(Y):
    need = Y.lib.yoco_gret_prefill_workspace_size(1, 100000, 1, 128, 128, 0, 1)
    assert need > 0
    st = Y.lib.yoco_gret_prefill_chunkwise(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, 1, 100000, 1, 128, 128, 0,
                                           1, 1, None, 0, None)
    assert st == Y.YOCO_ERR_WORKSPACE
    st = Y.lib.yoco_gret_prefill_chunkwise(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, 1, 100000, 1, 128, 128, 0,
                                           1, 1, ctypes.c_void_p(0x1010), need, None)
    assert st == Y.YOCO_ERR_WORKSPACE  # misaligned
    st = Y.lib.yoco_gret_prefill_chunkwise(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, 1, 100000, 1, 128, 128, 0,
                                           1, 1, ctypes.c_void_p(0x1000), need - 1, None)
    assert st == Y.YOCO_ERR_WORKSPACE  # too small


def test_gret_decode_rejects_bad_arguments(Y):
    L = Y.lib
    assert L.yoco_gret_decode_step(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, 1, 1, 32, 32, 1, 1, None) == \
        Y.YOCO_ERR_UNSUPPORTED
    assert L.yoco_gret_decode_step(None, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, 1, 1, 64, 64, 1, 1, None) == \
        Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_gret_decode_step(FAKE, FAKE, FAKE, FAKE, 16.0, ctypes.c_void_p(0x1004), FAKE, 1, 1, 64, 64, 1, 1,
                                   None) == Y.YOCO_ERR_INVALID_ARG


def _cache(Y, length=0, cap=16, d=64, Hkv=2, B=1, dtype=1):
    return Y._KVCacheC(0x2000, 0x3000, 0x4000, length, B, Hkv, d, cap, dtype)


def test_kv_append_capacity_and_validation(Y):
    L = Y.lib
    c = _cache(Y, length=14)
    need = L.yoco_shared_kv_workspace_size(1, 3, 64, ctypes.byref(c))
    st = L.yoco_shared_kv_project_append(FAKE, None, 1e-6, FAKE, FAKE, 3, 64, ctypes.byref(c), FAKE, need, None)
    assert st == Y.YOCO_ERR_CAPACITY
    assert c.len_host == 14  # unchanged
    assert b"capacity" in L.yoco_last_error()
    bad = _cache(Y, d=96)
    assert L.yoco_shared_kv_project_append(FAKE, None, 1e-6, FAKE, FAKE, 1, 64, ctypes.byref(bad), FAKE, 1 << 20,
                                           None) == Y.YOCO_ERR_UNSUPPORTED
    assert L.yoco_shared_kv_project_append(FAKE, None, -1.0, FAKE, FAKE, 1, 64, ctypes.byref(c), FAKE, 1 << 20,
                                           None) == Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_shared_kv_project_append(FAKE, None, 1e-6, FAKE, FAKE, 0, 64, ctypes.byref(c), FAKE, 1 << 20,
                                           None) == Y.YOCO_ERR_INVALID_ARG
    nolen = Y._KVCacheC(0x2000, 0x3000, 0, 0, 1, 2, 64, 16, 1)
    assert L.yoco_shared_kv_project_append(FAKE, None, 1e-6, FAKE, FAKE, 1, 64, ctypes.byref(nolen), FAKE, 1 << 20,
                                           None) == Y.YOCO_ERR_INVALID_ARG


def test_cross_attn_validation(Y):
    L = Y.lib
    c = _cache(Y, length=10)
    # rows past the cached length
    assert L.yoco_cross_attn_prefill(FAKE, 4, 3, 8, ctypes.byref(c), 0.1, FAKE, FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_cross_attn_prefill(FAKE, 4, 1, -1, ctypes.byref(c), 0.1, FAKE, FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_INVALID_ARG
    # Hq not a multiple of Hkv
    assert L.yoco_cross_attn_prefill(FAKE, 3, 1, 0, ctypes.byref(c), 0.1, FAKE, FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_UNSUPPORTED
    empty = _cache(Y, length=0)
    assert L.yoco_cross_attn_decode(FAKE, 4, ctypes.byref(empty), 0.1, 0, FAKE, FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_cross_attn_decode(FAKE, 4, ctypes.byref(c), 0.1, -2, FAKE, FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_INVALID_ARG
    big = _cache(Y, length=100000, cap=100000, Hkv=1)
    need = L.yoco_cross_attn_workspace_size(1, 4, 1, ctypes.byref(big), 0)
    assert need > 0
    assert L.yoco_cross_attn_decode(FAKE, 4, ctypes.byref(big), 0.1, 0, FAKE, None, 0, None) == \
        Y.YOCO_ERR_WORKSPACE


def test_kv_cache_bytes_match_teaching_numbers(Y):
    """Blog post Section 7: one shared K/V of 128 Ki tokens x 8 heads x 128 in
    2-byte elements is 0.5 GiB, whatever the number of cross layers."""
    assert Y.KVCache.nbytes(1, 8, 128, 131072, 2) == 2 ** 29


def test_selftest_rejects_bad_arguments(Y):
    L = Y.lib
    assert L.yoco_selftest_wait_timeout(ctypes.c_void_p(0x1010), 1000, None) == Y.YOCO_ERR_WORKSPACE
    assert L.yoco_selftest_wait_timeout(None, 1000, None) == Y.YOCO_ERR_WORKSPACE
    assert L.yoco_selftest_wait_timeout(FAKE, 0, None) == Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_selftest_wait_timeout(FAKE, 20_000_000_000, None) == Y.YOCO_ERR_INVALID_ARG


def _ring(Y, window=64, d=128, Hkv=2, B=1, dtype=1, pos=0):
    return Y._SwaRingC(0x2000, 0x3000, B, Hkv, d, window, pos, dtype)


def test_swa_validation(Y):
    L = Y.lib
    r = _ring(Y, pos=5)
    assert L.yoco_swa_prefill(FAKE, FAKE, FAKE, 4, 10, 0.1, FAKE, ctypes.byref(r), FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_INVALID_ARG  # prefill starts a sequence
    assert b"position" in L.yoco_last_error()
    r = _ring(Y, dtype=0)
    assert L.yoco_swa_prefill(FAKE, FAKE, FAKE, 4, 10, 0.1, FAKE, ctypes.byref(r), FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_UNSUPPORTED  # fp32 prefill
    r = _ring(Y, d=96)
    assert L.yoco_swa_decode(FAKE, FAKE, FAKE, 4, 0.1, FAKE, ctypes.byref(r), FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_UNSUPPORTED
    r = _ring(Y)
    assert L.yoco_swa_decode(FAKE, FAKE, FAKE, 3, 0.1, FAKE, ctypes.byref(r), FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_UNSUPPORTED  # Hq not a multiple of Hkv
    assert L.yoco_swa_decode(FAKE, FAKE, FAKE, 4, 0.1, FAKE, ctypes.byref(r), None, 0, None) == \
        Y.YOCO_ERR_WORKSPACE
    r = _ring(Y, window=0)
    assert L.yoco_swa_prefill(FAKE, FAKE, FAKE, 4, 10, 0.1, FAKE, ctypes.byref(r), FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_INVALID_ARG
    r = _ring(Y)
    assert L.yoco_swa_workspace_size(1, 4, ctypes.byref(r)) >= 256
    assert r.pos == 0  # failed calls do not move the ring


def test_group_norm_gate_validation(Y):
    L = Y.lib
    assert L.yoco_gret_group_norm_gate(FAKE, FAKE, None, None, 0.0, FAKE, 1, 4, 2, 128, 1, None) == \
        Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_gret_group_norm_gate(FAKE, FAKE, None, None, 1e-5, FAKE, 1, 4, 2, 96, 1, None) == \
        Y.YOCO_ERR_UNSUPPORTED
    assert L.yoco_gret_group_norm_gate(FAKE, None, None, None, 1e-5, FAKE, 1, 4, 2, 128, 1, None) == \
        Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_gret_group_norm_gate(FAKE, FAKE, None, None, 1e-5, FAKE, 1, 0, 2, 128, 1, None) == Y.YOCO_OK


def test_decode_step_gn_gate_validation(Y):
    L = Y.lib
    odd = ctypes.c_void_p(0x1004)  # 4-byte aligned only
    call = L.yoco_gret_decode_step_gn_gate
    assert call(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, None, None, 0.0, FAKE, 1, 2, 128, 128, 1, None) == \
        Y.YOCO_ERR_INVALID_ARG  # eps
    assert call(FAKE, FAKE, FAKE, FAKE, 0.0, FAKE, FAKE, None, None, 1e-5, FAKE, 1, 2, 128, 128, 1, None) == \
        Y.YOCO_ERR_INVALID_ARG  # tau
    assert call(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, None, None, None, 1e-5, FAKE, 1, 2, 128, 128, 1, None) == \
        Y.YOCO_ERR_INVALID_ARG  # gate
    assert call(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, None, None, 1e-5, FAKE, 1, 2, 96, 96, 1, None) == \
        Y.YOCO_ERR_UNSUPPORTED
    assert call(FAKE, FAKE, FAKE, FAKE, 16.0, odd, FAKE, None, None, 1e-5, FAKE, 1, 2, 128, 128, 1, None) == \
        Y.YOCO_ERR_INVALID_ARG  # state alignment


def test_rope_validation(Y):
    L = Y.lib
    assert L.yoco_rope_apply(FAKE, 1, 4, 2, 128, 0, 1.0, 1, None) == Y.YOCO_ERR_INVALID_ARG  # base must exceed 1
    assert L.yoco_rope_apply(FAKE, 1, 4, 2, 96, 0, 1e4, 1, None) == Y.YOCO_ERR_UNSUPPORTED
    assert L.yoco_rope_apply(FAKE, 1, 4, 2, 128, -1, 1e4, 1, None) == Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_rope_apply(FAKE, 1, 0, 2, 128, 0, 1e4, 1, None) == Y.YOCO_OK  # nothing to do
    c = _cache(Y, length=10)
    c.rope_base = -5.0
    assert L.yoco_cross_attn_decode(FAKE, 4, ctypes.byref(c), 0.1, 0, FAKE, FAKE, 1 << 20, None) == \
        Y.YOCO_ERR_INVALID_ARG
    assert b"rope_base" in L.yoco_last_error()


def test_qkvg_validation(Y):
    L = Y.lib
    args = lambda H, d, rb=0.0, ws=FAKE, n=1 << 20: (FAKE, FAKE, 1, 64, 256, H, d, 0, rb, FAKE, FAKE, FAKE, FAKE,  # noqa: E731
                                                    ws, n, None)
    assert L.yoco_gret_qkvg_project(*args(12, 128)) == Y.YOCO_ERR_UNSUPPORTED  # H not a multiple of 8
    assert L.yoco_gret_qkvg_project(*args(8, 96)) == Y.YOCO_ERR_UNSUPPORTED
    assert L.yoco_gret_qkvg_project(*args(8, 128, rb=-1.0)) == Y.YOCO_ERR_INVALID_ARG
    assert L.yoco_gret_qkvg_project(*args(8, 128, rb=1e4, ws=None, n=0)) == Y.YOCO_ERR_WORKSPACE
    assert L.yoco_gret_qkvg_workspace_size(1, 64, 8, 128, 1e4) == 256 + 64 * 64 * 8


def test_test_hook_rejects_unknown_hooks_and_ranges(Y):
    assert Y.lib.yoco_test_hook(0, 1) == Y.YOCO_ERR_INVALID_ARG
    assert Y.lib.yoco_test_hook(99, 1) == Y.YOCO_ERR_INVALID_ARG
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_FAIL_NEXT_CALLS, -1) == Y.YOCO_ERR_INVALID_ARG
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_FAIL_NEXT_CALLS, 10 ** 7) == Y.YOCO_ERR_INVALID_ARG
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_GRET_SEG0_DELAY_NS, 2 * 10 ** 9) == Y.YOCO_ERR_INVALID_ARG
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_GRET_SEG0_DELAY_NS, 0) == Y.YOCO_OK


def test_injected_launch_failure_comes_after_argument_checks(Y):
    """An injected failure is returned as YOCO_ERR_CUDA by calls whose arguments
    pass, one per call, before anything is enqueued; a call that fails its
    argument checks reports that instead and leaves the injection pending."""
    def decode_step(B=1):
        return Y.lib.yoco_gret_decode_step(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, B, 2, 64, 64, 0, 0, None)

    n0 = Y.lib.yoco_launch_count()
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_FAIL_NEXT_CALLS, 2) == Y.YOCO_OK
    try:
        assert decode_step() == Y.YOCO_ERR_CUDA
        assert b"launch failure" in Y.lib.yoco_last_error()
        assert decode_step(B=0) == Y.YOCO_ERR_INVALID_ARG  # argument error first; injection still pending
        assert Y.lib.yoco_gret_prefill_chunkwise(FAKE, FAKE, FAKE, FAKE, 16.0, FAKE, FAKE, 1, 8, 1, 64, 64, 0, 0, 0,
                                                 FAKE, 1 << 20, None) == Y.YOCO_ERR_CUDA
        assert b"launch failure" in Y.lib.yoco_last_error()
        assert Y.lib.yoco_launch_count() == n0  # nothing was enqueued
    finally:
        assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_FAIL_NEXT_CALLS, 0) == Y.YOCO_OK


def test_every_documented_chunk_value_is_accepted(Y):
    """The header documents chunk in {0, 64, 128}: those pass the argument checks
    (the call then asks for its workspace or, needing none, tries to launch,
    which fails without a GPU), every other value is refused."""
    header = open(HEADER).read()
    assert "chunk        0, 64 or 128" in header
    # an accepted call must not reach a launch with these fake pointers, even where
    # a GPU is present: injected failures stand in for every launch meanwhile
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_FAIL_NEXT_CALLS, 1000) == Y.YOCO_OK
    try:
        for dt, d in ((1, 128), (1, 64), (0, 64)):
            for chunk in (0, 64, 128):
                st = _prefill(Y, dk=d, dv=d, in_dt=dt, out_dt=dt, chunk=chunk)
                assert st in (Y.YOCO_ERR_WORKSPACE, Y.YOCO_ERR_CUDA), (dt, d, chunk, st)
            for chunk in (1, 16, 32, 96, 256):
                st = _prefill(Y, dk=d, dv=d, in_dt=dt, out_dt=dt, chunk=chunk)
                assert st == Y.YOCO_ERR_UNSUPPORTED, (dt, d, chunk)
    finally:
        assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_FAIL_NEXT_CALLS, 0) == Y.YOCO_OK


def test_selftest_occupy_rejects_bad_arguments(Y):
    assert Y.lib.yoco_selftest_occupy_sms(0, 1000, None) == Y.YOCO_ERR_INVALID_ARG
    assert Y.lib.yoco_selftest_occupy_sms(10, 0, None) == Y.YOCO_ERR_INVALID_ARG
    assert Y.lib.yoco_selftest_occupy_sms(10, 2 * 10 ** 9, None) == Y.YOCO_ERR_INVALID_ARG


def test_release_build_reports_no_debug_checks(Y):
    """yoco_debug_checks answers without touching a device: a release build
    has no index checks compiled in."""
    if os.environ.get("YOCO_LIB_PATH"):
        pytest.skip("this process runs another build")
    w = ctypes.c_uint32(7)
    assert Y.lib.yoco_debug_checks(0, ctypes.byref(w)) == Y.YOCO_ERR_UNSUPPORTED
    assert w.value == 0
    assert Y.lib.yoco_debug_checks(0, None) == Y.YOCO_ERR_INVALID_ARG
