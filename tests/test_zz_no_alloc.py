"""The allocation-free decode entry point (collected last on purpose).

yoco_cross_attn_decode_noalloc serves callers that cannot allocate device
memory while they decode; it keeps its split partials in scratch built into
the library instead of a caller workspace.  Its output must match
yoco_cross_attn_decode's on the same inputs, on consecutive calls (the
scratch keeps the previous call's contents), and an explicit split count
whose partials do not fit must be refused before anything runs.
"""
import ctypes

import numpy as np
import pytest

import synth
from _util import gen, host_f64, rel_l2

pytestmark = pytest.mark.gpu

BF16_REL_L2 = 1e-2
SEED = synth.DEFAULT_SEED


@pytest.fixture(scope="module")
def Y():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import gated_retention_shared_gb300 as Y
    return Y


def _cache(Y, B, Hkv, d, length):
    _, Kd = gen(SEED, synth.stream_id(40, 0, synth.T_CACHE_K), (B, Hkv, length, d), "bf16")
    _, Vd = gen(SEED, synth.stream_id(40, 0, synth.T_CACHE_V), (B, Hkv, length, d), "bf16")
    cache = Y.KVCache(B, Hkv, d, length, dtype=Kd.dtype, k=Kd, v=Vd)
    cache.set_length(length)
    return cache


@pytest.mark.parametrize("num_splits", [0, 5])
def test_noalloc_decode_matches_workspace_decode_twice(Y, num_splits):
    import torch
    B, Hq, Hkv, d, length = 2, 24, 8, 128, 3001
    cache = _cache(Y, B, Hkv, d, length)
    for call in range(2):  # two calls in a row, different queries
        _, Qd = gen(SEED, synth.stream_id(40, 1, synth.T_QX, call), (B, Hq, d), "bf16")
        O_ref = torch.empty_like(Qd)
        Y.yoco_cross_attn_decode(Qd, cache, O_ref, num_splits=num_splits)
        O = torch.full_like(Qd, float("nan"))
        st = Y.lib.yoco_cross_attn_decode_noalloc(ctypes.c_void_p(Qd.data_ptr()), Hq, ctypes.byref(cache.c),
                                                  d ** -0.5, num_splits, ctypes.c_void_p(O.data_ptr()),
                                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == Y.YOCO_OK, Y.lib.yoco_last_error()
        torch.cuda.synchronize()
        assert np.isfinite(host_f64(O)).all()
        assert rel_l2(host_f64(O), host_f64(O_ref)) <= BF16_REL_L2


def test_noalloc_decode_refuses_oversized_split_count(Y):
    import torch
    B, Hq, Hkv, d, length = 2, 24, 8, 128, 3001
    cache = _cache(Y, B, Hkv, d, length)
    Qd = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    O = torch.zeros_like(Qd)
    st = Y.lib.yoco_cross_attn_decode_noalloc(ctypes.c_void_p(Qd.data_ptr()), Hq, ctypes.byref(cache.c), 0.1,
                                              4096, ctypes.c_void_p(O.data_ptr()), None)
    assert st == Y.YOCO_ERR_UNSUPPORTED
    assert b"scratch" in Y.lib.yoco_last_error()
    torch.cuda.synchronize()
    assert bool((O == 0).all())


def test_noalloc_decode_refuses_more_than_4096_splits(Y):
    """The merge holds one factor per split, at most 4096; a count above that
    is refused even when its partials would fit the scratch."""
    import torch
    B, Hq, Hkv, d, length = 1, 1, 1, 64, 3001
    cache = _cache(Y, B, Hkv, d, length)
    Qd = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    O = torch.zeros_like(Qd)
    st = Y.lib.yoco_cross_attn_decode_noalloc(ctypes.c_void_p(Qd.data_ptr()), Hq, ctypes.byref(cache.c), 0.1,
                                              5000, ctypes.c_void_p(O.data_ptr()), None)
    assert st == Y.YOCO_ERR_UNSUPPORTED
    assert b"4096" in Y.lib.yoco_last_error()
    torch.cuda.synchronize()
    assert bool((O == 0).all())
